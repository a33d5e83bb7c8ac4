// api.cu — C ABI of the decode megakernel (declared in include/mk.h).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/mk.h"
#include "mk_kernel.h"
#include "planner.h"
#include "ptx.cuh"

using namespace mk;

struct mk_plan {
    mk_model_cfg cfg;
    mk_plan_options opt;
    // test_poison_scratch: the (address, bytes) ranges of activation scratch
    // filled with 0xFF (NaN as fp32 and as bf16) before every step
    std::vector<std::pair<void *, size_t>> poison;
    PlanTables tables;
    int device = 0;
    int variant = 0;
    size_t smem = 0;
    CtlLayout cl{};
    // device memory owned by the plan
    std::vector<void *> allocs;
    LayerW *d_layers = nullptr;
    Task *d_tasks = nullptr;
    int32_t *d_queue = nullptr;
    float *d_x = nullptr, *d_qkv = nullptr, *d_part = nullptr, *d_attn = nullptr, *d_h = nullptr;
    float2 *d_rope = nullptr;
    uint32_t *d_ctl = nullptr;
    int32_t *d_iota = nullptr;       // 0..max_seq-1, positions of prefill steps
    int32_t *d_stage_tok = nullptr;  // staging for the host-buffer entry point
    int32_t *d_stage_pos = nullptr;
    float *d_stage_logits = nullptr;
    uint32_t *h_err = nullptr;       // pinned host copy of the device error word
    uint64_t *d_trace = nullptr;
    int32_t trace_stride = 0;
    // batched path
    uint16_t *d_xa = nullptr, *d_attn_a = nullptr, *d_h_a = nullptr;
    float *d_ssq = nullptr, *d_tc_part = nullptr;
    uint8_t *d_tmaps = nullptr;
    uint8_t *d_down_maps = nullptr;  // batch 1: per-layer w_down tensor maps
    KParams base{};
    // host copies of the weight pointers (the chunked-prefill engine's plan reuses them)
    std::vector<LayerW> hlw;
    const void *w_embed = nullptr, *w_lm = nullptr, *w_final = nullptr;
    // chunked-prefill engine, made on first use: a kv-append plan whose
    // kPrefillRows batch rows are consecutive tokens of one sequence
    mk_plan *pre = nullptr;
    int32_t *d_stage_off = nullptr;  // dynamic dispatch: first task of each stage
    float *d_pre_logits = nullptr;  // [kPrefillRows][vocab]
    int32_t *d_pre_tok = nullptr, *d_pre_pos = nullptr;
    // tensor maps of the last KV cache seen (encoded once per cache, not per step)
    mk_kv_cache kv_seen{};
    bool kv_maps_valid = false;
    alignas(64) uint8_t kv_maps[2][128];
    int32_t kv_halves_3d = 0;
};

namespace mk {

// cuTensorMapEncodeTiled from the driver, looked up once (no libcuda link).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    }
    return fn;
}

// Row-major bf16 [outer][inner] matrix read in boxes of 64 columns x
// box_outer rows, 128-byte swizzled (the tcgen05 K-major operand layout).
// Rows and columns past the end read as zero.
bool encode_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcTileK, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A pool of d = 128 as a 3-D view (column within a 64-column half, token
// row, half): one box of 64 columns x ts tokens x 2 halves lands in shared
// memory as the two 128-byte-swizzled half tiles one after the other, the
// layout two 2-D copies would give, in one copy.
bool encode_kv_halves(CUtensorMap *m, const void *base, uint64_t rows, uint32_t ts) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {64, rows, 2};
    const cuuint64_t strides[2] = {256, 128};
    const cuuint32_t box[3] = {64, ts, 2};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K and V pools as [L * num_pages * nkv * page_size][d] bf16 rows, read in
// boxes of 64 columns x ts tokens (d = 64), or of both halves of d = 128 at
// once where the driver takes the 3-D view (kv_halves_3d), else per half.
bool encode_kv_maps(KParams &k, const mk_model_cfg &c, const mk_kv_cache &kv, int32_t ts) {
    const uint64_t rows = (uint64_t)c.n_layers * kv.num_pages * c.n_kv_heads * c.page_size;
    if (rows >= (1ull << 31)) return false;
    k.kv_halves_3d = 0;
    if (c.head_dim == 128 &&
        encode_kv_halves(reinterpret_cast<CUtensorMap *>(k.kv_maps[0]), kv.k_pool, rows, (uint32_t)ts) &&
        encode_kv_halves(reinterpret_cast<CUtensorMap *>(k.kv_maps[1]), kv.v_pool, rows, (uint32_t)ts)) {
        k.kv_halves_3d = 1;
        return true;
    }
    return encode_bf16_2d(reinterpret_cast<CUtensorMap *>(k.kv_maps[0]), kv.k_pool, c.head_dim, rows, ts) &&
           encode_bf16_2d(reinterpret_cast<CUtensorMap *>(k.kv_maps[1]), kv.v_pool, c.head_dim, rows, ts);
}

bool down_tma_ok(const MvGeom &g) {
    return g.rps == 0 && g.row_mult == 1 && g.kc == 2048 && g.K % g.kc == 0 && g.ksplit > 2 && g.rpp >= 1 &&
           g.rpp <= 8;
}

// w_down [rows][K] bf16 seen as [rows][K/256][256]: a box of rpp rows x
// kc/256 blocks x 256 columns lands in shared memory as rpp rows of kc
// columns, row r at byte offset r * kc * 2 (the bulk copies' slot layout).
// Rows past the end read as zero.
bool encode_down_map(void *m, const void *w_down, const MvGeom &g) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || !down_tma_ok(g)) return false;
    const cuuint64_t dims[3] = {256, (cuuint64_t)g.K / 256, (cuuint64_t)g.rows};
    const cuuint64_t strides[2] = {512, (cuuint64_t)g.K * 2};
    const cuuint32_t box[3] = {256, (cuuint32_t)g.kc / 256, (cuuint32_t)g.rpp};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(reinterpret_cast<CUtensorMap *>(m), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(w_down),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mk

namespace {

template <typename T>
mk_status dev_alloc(mk_plan *p, T **ptr, size_t count) {
    void *q = nullptr;
    if (cudaMalloc(&q, std::max<size_t>(count, 1) * sizeof(T)) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_OOM;
    }
    p->allocs.push_back(q);
    *ptr = static_cast<T *>(q);
    return MK_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mk_status check_weights(const mk_model_cfg &c, const mk_weight_ptrs *w) {
    if (!w) return MK_ERR_INVALID;
    if (!aligned16(w->embed) || !aligned16(w->lm_head) || !aligned16(w->final_norm)) return MK_ERR_INVALID;
    if (c.tied_embeddings && w->lm_head != w->embed) return MK_ERR_INVALID;
    const void *const *arrs[] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->w_gate, w->w_up, w->w_down};
    for (const void *const *a : arrs) {
        if (!a) return MK_ERR_INVALID;
        for (int l = 0; l < c.n_layers; ++l)
            if (!aligned16(a[l])) return MK_ERR_INVALID;
    }
    return MK_OK;
}

// Validates the cache and keeps its two tensor maps in the plan: they are
// encoded again only when the pools or their page counts change.
mk_status check_kv(mk_plan *p, const mk_kv_cache *kv) {
    if (!kv || !aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !aligned16(kv->page_table)) return MK_ERR_INVALID;
    if (kv->num_pages <= 0 || kv->max_pages_per_seq <= 0) return MK_ERR_INVALID;
    if ((int64_t)kv->max_pages_per_seq * p->cfg.page_size < p->cfg.max_seq) return MK_ERR_INVALID;
    const mk_kv_cache &s = p->kv_seen;
    if (p->kv_maps_valid && s.k_pool == kv->k_pool && s.v_pool == kv->v_pool && s.num_pages == kv->num_pages)
        return MK_OK;
    KParams probe{};
    p->kv_maps_valid = false;
    if (!encode_kv_maps(probe, p->cfg, *kv, p->tables.g.tps)) return MK_ERR_INVALID;  // pools too large for a map
    std::memcpy(p->kv_maps, probe.kv_maps, sizeof(p->kv_maps));
    p->kv_halves_3d = probe.kv_halves_3d;
    p->kv_seen = *kv;
    p->kv_maps_valid = true;
    return MK_OK;
}

mk_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MK_OK;
    cudaGetLastError();
    if (e == cudaErrorCooperativeLaunchTooLarge) return MK_ERR_LAUNCH;
    return MK_ERR_CUDA;
}

void free_plan(mk_plan *p) {
    if (p->pre) free_plan(p->pre);
    if (p->h_err) cudaFreeHost(p->h_err);
    for (void *q : p->allocs) cudaFree(q);
    p->allocs.clear();
    delete p;
}

KParams step_params(const mk_plan *p, const int32_t *tokens, int32_t tok_stride, const int32_t *positions,
                    int32_t pos_stride, const mk_kv_cache *kv, float *logits) {
    KParams k = p->base;
    std::memcpy(k.kv_maps, p->kv_maps, sizeof(k.kv_maps));  // encoded by check_kv
    k.kv_halves_3d = p->kv_halves_3d;
    k.k_pool = static_cast<uint16_t *>(kv->k_pool);
    k.v_pool = static_cast<uint16_t *>(kv->v_pool);
    k.page_table = kv->page_table;
    k.num_pages = kv->num_pages;
    k.max_pages = kv->max_pages_per_seq;
    k.pt_stride = kv->max_pages_per_seq;
    k.tokens = tokens;
    k.tok_stride = tok_stride;
    k.positions = positions;
    k.pos_stride = pos_stride;
    k.logits = logits;
    return k;
}

mk_status clear_trace(mk_plan *p, cudaStream_t s) {
    if (!p->d_trace) return MK_OK;
    return cuda_status(
        cudaMemsetAsync(p->d_trace, 0, (size_t)p->tables.g.num_ctas * p->trace_stride * 8 * sizeof(uint64_t), s));
}

// test_poison_scratch: NaN-fill the activation scratch before a step.
mk_status poison_scratch(mk_plan *p, cudaStream_t s) {
    for (const auto &r : p->poison)
        if (cudaMemsetAsync(r.first, 0xFF, r.second, s) != cudaSuccess) return cuda_status(cudaGetLastError());
    return MK_OK;
}

mk_status launch_step(mk_plan *p, const KParams &k, cudaStream_t s) {
    cudaError_t e = cudaSetDevice(p->device);
    if (e != cudaSuccess) return cuda_status(e);
    mk_status st = clear_trace(p, s);
    if (st != MK_OK) return st;
    if ((st = poison_scratch(p, s)) != MK_OK) return st;
    return cuda_status(launch_megakernel(k, p->variant, p->tables.g.num_ctas, p->smem, true, s));
}

}  // namespace

extern "C" {

const char *mk_status_string(mk_status s) {
    switch (s) {
        case MK_OK: return "ok";
        case MK_ERR_INVALID: return "invalid argument";
        case MK_ERR_CUDA: return "CUDA runtime error";
        case MK_ERR_LAUNCH: return "cooperative grid cannot be co-resident";
        case MK_ERR_TIMEOUT: return "device wait exceeded the time budget";
        case MK_ERR_BOUNDS: return "token, position or page id out of range";
        case MK_ERR_OOM: return "out of device memory";
        case MK_ERR_UNSUPPORTED: return "unsupported shape";
    }
    return "unknown status";
}

const char *mk_error_site_string(int32_t site) {
    switch (site) {
        case SITE_NONE: return "none";
        case SITE_EVENT_WAIT: return "scheduler event-counter wait";
        case SITE_READY_WAIT: return "compute wait for task release";
        case SITE_FULL_WAIT: return "compute wait for a filled ring slot";
        case SITE_EMPTY_WAIT: return "producer wait for a free ring slot";
        case SITE_DRAIN_WAIT: return "producer drain of copies in flight";
        case SITE_TOKEN: return "token id out of range";
        case SITE_POSITION: return "position out of range";
        case SITE_PAGE: return "page id out of range";
        case SITE_ABORTED: return "aborted";
    }
    return "unknown site";
}

mk_status mk_plan_describe(const mk_model_cfg *cfg, const mk_plan_options *opt, int32_t num_ctas,
                           mk_task_info *out, int32_t capacity, int32_t *n_tasks, int32_t *n_events) {
    if (!cfg || num_ctas <= 0 || !n_tasks || !n_events) return MK_ERR_INVALID;
    mk_plan_options o = resolve_options(*cfg, opt, num_ctas);
    PlanTables t;
    mk_status st = build_plan(*cfg, o, &t);
    if (st != MK_OK) return st;
    *n_tasks = (int32_t)t.tasks.size();
    *n_events = t.g.n_events;
    if (capacity < *n_tasks || (!out && *n_tasks > 0)) return MK_ERR_INVALID;
    for (int32_t c = 0; c < o.num_ctas; ++c)
        for (int32_t i = (t.g.jit ? (c == 0 ? 0 : *n_tasks) : t.queue_off[c]);
             i < (t.g.jit ? (c == 0 ? *n_tasks : 0) : t.queue_off[c + 1]); ++i) {
            const Task &k = t.tasks[i];
            mk_task_info &d = out[i];
            d.cta = t.g.jit ? -1 : c;  // dynamic dispatch: claimed at run time, stage by stage
            d.op = k.op;
            d.layer = k.layer;
            d.wait_event = k.wait_ev == kNoEvent ? -1 : k.wait_ev;
            d.wait_count = (int32_t)k.wait_count;
            d.signal_event = k.signal_ev == kNoEvent ? -1 : k.signal_ev;
            d.a0 = k.a0;
            d.a1 = k.a1;
            d.a2 = k.a2;
            d.a3 = k.a3;
        }
    return MK_OK;
}

mk_status mk_plan_create_ex(const mk_model_cfg *cfg, const mk_weight_ptrs *w, const mk_plan_options *opt,
                            mk_plan **out) {
    if (!cfg || !out) return MK_ERR_INVALID;
    *out = nullptr;
    mk_status st = check_cfg(*cfg);
    if (st != MK_OK) return st;
    if ((st = check_weights(*cfg, w)) != MK_OK) return st;

    int dev = 0, sms = 0, smem_optin = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) {
        cudaGetLastError();
        return MK_ERR_CUDA;
    }
    if (!coop) return MK_ERR_UNSUPPORTED;

    mk_plan *p = new (std::nothrow) mk_plan();
    if (!p) return MK_ERR_OOM;
    p->cfg = *cfg;
    p->device = dev;
    p->opt = resolve_options(*cfg, opt, sms);
    if (p->opt.num_slots > kMaxSlots) p->opt.num_slots = kMaxSlots;
    if ((st = build_plan(*cfg, p->opt, &p->tables)) != MK_OK) {
        free_plan(p);
        return st;
    }
    PlanGeom &g = p->tables.g;
    if (g.tc && g.num_slots == 0) {
        // as many weight tiles in flight as shared memory holds
        const size_t fixed = megakernel_smem_bytes(0, 0, g.aslot_bytes, g.num_aslots);
        g.num_slots = (int32_t)std::min<size_t>(kMaxSlots, ((size_t)smem_optin - fixed) / g.slot_bytes);
        p->opt.num_slots = g.num_slots;
        if (g.num_slots < 2) {
            free_plan(p);
            return MK_ERR_UNSUPPORTED;
        }
    }
    p->smem = megakernel_smem_bytes(g.slot_bytes, g.num_slots, g.tc ? g.aslot_bytes : 0, g.tc ? g.num_aslots : 0);
    if ((int)p->smem > smem_optin) {
        free_plan(p);
        return MK_ERR_INVALID;
    }
    const int32_t max_k = std::max({cfg->hidden, cfg->ffn_dim, cfg->n_q_heads * cfg->head_dim});
    p->variant = megakernel_variant(max_k, g.tc, g.jit);
    if (megakernel_set_smem(p->variant, p->smem) != cudaSuccess) {
        cudaGetLastError();
        free_plan(p);
        return MK_ERR_CUDA;
    }
    int per_sm = 0;
    if (megakernel_max_active(p->variant, p->smem, &per_sm) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        free_plan(p);
        return MK_ERR_LAUNCH;
    }

    const mk_model_cfg &c = *cfg;
    const int32_t G = c.n_q_heads / c.n_kv_heads, S = g.attn_splits;
    const int32_t qkv_rows = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    const int32_t n_stages = g.jit ? (int32_t)p->tables.stage_off.size() - 1 : 0;
    p->cl = ctl_layout(g.n_events, c.batch * c.n_kv_heads, g.tc ? g.n_tile_ctrs : 0, c.batch, n_stages);
    const size_t n_part = (size_t)c.batch * c.n_kv_heads * S * G * (c.head_dim + 2);
    if ((st = dev_alloc(p, &p->d_layers, c.n_layers)) || (st = dev_alloc(p, &p->d_tasks, p->tables.tasks.size())) ||
        (st = dev_alloc(p, &p->d_queue, p->tables.queue_off.size())) ||
        (st = dev_alloc(p, &p->d_x, (size_t)c.batch * c.hidden)) ||
        (st = dev_alloc(p, &p->d_qkv, (size_t)c.batch * qkv_rows)) || (st = dev_alloc(p, &p->d_part, n_part)) ||
        (st = dev_alloc(p, &p->d_attn, (size_t)c.batch * c.n_q_heads * c.head_dim)) ||
        (st = dev_alloc(p, &p->d_h, (size_t)c.batch * c.ffn_dim)) ||
        (st = dev_alloc(p, &p->d_rope, (size_t)c.max_seq * (c.head_dim / 2))) ||
        (st = dev_alloc(p, &p->d_ctl, (size_t)p->cl.total)) || (st = dev_alloc(p, &p->d_iota, (size_t)c.max_seq)) ||
        (st = dev_alloc(p, &p->d_stage_tok, (size_t)c.batch)) || (st = dev_alloc(p, &p->d_stage_pos, (size_t)c.batch)) ||
        (st = dev_alloc(p, &p->d_stage_logits, (size_t)c.batch * c.vocab))) {
        free_plan(p);
        return st;
    }
    if (g.jit) {
        if ((st = dev_alloc(p, &p->d_stage_off, p->tables.stage_off.size())) != MK_OK) {
            free_plan(p);
            return st;
        }
        if (cudaMemcpy(p->d_stage_off, p->tables.stage_off.data(), p->tables.stage_off.size() * sizeof(int32_t),
                       cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            free_plan(p);
            return MK_ERR_CUDA;
        }
    }
    if (cudaHostAlloc(reinterpret_cast<void **>(&p->h_err), 4 * sizeof(uint32_t), cudaHostAllocDefault) !=
        cudaSuccess) {
        cudaGetLastError();
        p->h_err = nullptr;
        free_plan(p);
        return MK_ERR_OOM;
    }
    const int32_t n_tmaps = c.n_layers * 7 + 4;
    if (g.tc) {
        const size_t part = (size_t)g.num_ctas * 2 * 2 * g.npad * kTcTileM;
        const size_t rows2 = 2 * (size_t)g.npad;  // split-bf16 operands: high parts, then low parts
        if ((st = dev_alloc(p, &p->d_xa, rows2 * c.hidden)) ||
            (st = dev_alloc(p, &p->d_attn_a, rows2 * c.n_q_heads * c.head_dim)) ||
            (st = dev_alloc(p, &p->d_h_a, rows2 * c.ffn_dim)) ||
            (st = dev_alloc(p, &p->d_ssq, (size_t)c.batch * g.h_tiles)) || (st = dev_alloc(p, &p->d_tc_part, part)) ||
            (st = dev_alloc(p, &p->d_tmaps, (size_t)n_tmaps * sizeof(CUtensorMap)))) {
            free_plan(p);
            return st;
        }
    }
    if (!g.tc && down_tma_ok(g.mv[OP_DOWN])) {
        // one TMA copy per down-projection slot instead of one bulk copy per row
        std::vector<CUtensorMap> dm(c.n_layers);
        bool ok = true;
        for (int l = 0; l < c.n_layers && ok; ++l) ok = encode_down_map(&dm[l], w->w_down[l], g.mv[OP_DOWN]);
        if (ok) {
            if ((st = dev_alloc(p, &p->d_down_maps, dm.size() * sizeof(CUtensorMap))) != MK_OK) {
                free_plan(p);
                return st;
            }
            if (cudaMemcpy(p->d_down_maps, dm.data(), dm.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) !=
                cudaSuccess) {
                cudaGetLastError();
                free_plan(p);
                return MK_ERR_CUDA;
            }
        }
    }
    if (p->opt.trace) {
        for (int32_t i = 0; i < g.num_ctas; ++i)
            p->trace_stride = std::max(p->trace_stride, p->tables.queue_off[i + 1] - p->tables.queue_off[i]);
        if ((st = dev_alloc(p, &p->d_trace, (size_t)g.num_ctas * p->trace_stride * 8)) != MK_OK) {
            free_plan(p);
            return st;
        }
    }

    p->w_embed = w->embed;
    p->w_lm = w->lm_head;
    p->w_final = w->final_norm;
    std::vector<LayerW> &lw = p->hlw;
    lw.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        lw[l].attn_norm = static_cast<const uint16_t *>(w->attn_norm[l]);
        lw[l].wq = static_cast<const uint16_t *>(w->wq[l]);
        lw[l].wk = static_cast<const uint16_t *>(w->wk[l]);
        lw[l].wv = static_cast<const uint16_t *>(w->wv[l]);
        lw[l].wo = static_cast<const uint16_t *>(w->wo[l]);
        lw[l].mlp_norm = static_cast<const uint16_t *>(w->mlp_norm[l]);
        lw[l].w_gate = static_cast<const uint16_t *>(w->w_gate[l]);
        lw[l].w_up = static_cast<const uint16_t *>(w->w_up[l]);
        lw[l].w_down = static_cast<const uint16_t *>(w->w_down[l]);
    }
    std::vector<int32_t> iota(c.max_seq);
    for (int32_t i = 0; i < c.max_seq; ++i) iota[i] = i;
    cudaError_t e = cudaMemcpy(p->d_layers, lw.data(), lw.size() * sizeof(LayerW), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemcpy(p->d_tasks, p->tables.tasks.data(), p->tables.tasks.size() * sizeof(Task),
                       cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemcpy(p->d_queue, p->tables.queue_off.data(), p->tables.queue_off.size() * sizeof(int32_t),
                       cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(p->d_iota, iota.data(), iota.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && g.tc) {
        // tensor maps of every weight matrix (128-row boxes) and of the three
        // activation operands (npad-row boxes; rows past the batch read as 0)
        const int32_t H = c.hidden, I = c.ffn_dim, qd = c.n_q_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim;
        std::vector<CUtensorMap> maps(n_tmaps);
        bool ok = true;
        for (int l = 0; l < c.n_layers && ok; ++l) {
            CUtensorMap *m = &maps[(size_t)l * 7];
            ok = encode_bf16_2d(m + 0, w->wq[l], H, qd, kTcTileM) && encode_bf16_2d(m + 1, w->wk[l], H, kd, kTcTileM) &&
                 encode_bf16_2d(m + 2, w->wv[l], H, kd, kTcTileM) && encode_bf16_2d(m + 3, w->wo[l], qd, H, kTcTileM) &&
                 encode_bf16_2d(m + 4, w->w_gate[l], H, I, kTcTileM) &&
                 encode_bf16_2d(m + 5, w->w_up[l], H, I, kTcTileM) && encode_bf16_2d(m + 6, w->w_down[l], I, H, kTcTileM);
        }
        CUtensorMap *m = &maps[(size_t)c.n_layers * 7];
        ok = ok && encode_bf16_2d(m + 0, w->lm_head, H, c.vocab, kTcTileM) &&
             encode_bf16_2d(m + 1, p->d_xa, H, 2 * g.npad, 2 * g.npad) &&
             encode_bf16_2d(m + 2, p->d_attn_a, qd, 2 * g.npad, 2 * g.npad) &&
             encode_bf16_2d(m + 3, p->d_h_a, I, 2 * g.npad, 2 * g.npad);
        if (!ok) {
            free_plan(p);
            return MK_ERR_CUDA;
        }
        e = cudaMemcpy(p->d_tmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
        // padding rows (sequences past the batch) stay zero
        if (e == cudaSuccess) e = cudaMemset(p->d_xa, 0, 2 * (size_t)g.npad * c.hidden * 2);
        if (e == cudaSuccess) e = cudaMemset(p->d_attn_a, 0, 2 * (size_t)g.npad * qd * 2);
        if (e == cudaSuccess) e = cudaMemset(p->d_h_a, 0, 2 * (size_t)g.npad * I * 2);
    }
    if (e == cudaSuccess) e = cudaMemset(p->d_ctl, 0, (size_t)p->cl.total * sizeof(uint32_t));
    if (e == cudaSuccess) e = launch_rope_table(p->d_rope, c.max_seq, c.head_dim, c.rope_theta, 0);
    if (p->opt.test_poison_scratch) {
        // every buffer a step writes before it reads; the split-bf16 operands
        // only in their batch rows (high and low parts), the padding rows
        // must stay zero
        const size_t B = (size_t)c.batch;
        auto add = [&](void *q, size_t bytes) { p->poison.emplace_back(q, bytes); };
        add(p->d_x, B * c.hidden * 4);
        add(p->d_qkv, B * qkv_rows * 4);
        add(p->d_part, n_part * 4);
        add(p->d_attn, B * c.n_q_heads * c.head_dim * 4);
        add(p->d_h, B * c.ffn_dim * 4);
        if (g.tc) {
            const size_t qd = (size_t)c.n_q_heads * c.head_dim;
            const size_t widths[3] = {(size_t)c.hidden, qd, (size_t)c.ffn_dim};
            uint16_t *bufs[3] = {p->d_xa, p->d_attn_a, p->d_h_a};
            for (int i = 0; i < 3; ++i) {
                add(bufs[i], B * widths[i] * 2);
                add(bufs[i] + (size_t)g.npad * widths[i], B * widths[i] * 2);
            }
            add(p->d_ssq, B * g.h_tiles * 4);
            add(p->d_tc_part, (size_t)g.num_ctas * 2 * 2 * g.npad * kTcTileM * 4);
        }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaGetLastError();
        free_plan(p);
        return MK_ERR_CUDA;
    }

    KParams &k = p->base;
    k.L = c.n_layers;
    k.H = c.hidden;
    k.nq = c.n_q_heads;
    k.nkv = c.n_kv_heads;
    k.d = c.head_dim;
    k.I = c.ffn_dim;
    k.V = c.vocab;
    k.B = c.batch;
    k.max_seq = c.max_seq;
    k.page_size = c.page_size;
    k.eps = c.rms_eps;
    k.qkv_rows = qkv_rows;
    k.embed = static_cast<const uint16_t *>(w->embed);
    k.lm_head = static_cast<const uint16_t *>(w->lm_head);
    k.final_norm = static_cast<const uint16_t *>(w->final_norm);
    k.layers = p->d_layers;
    k.x = p->d_x;
    k.qkv = p->d_qkv;
    k.attn_part = p->d_part;
    k.attn_out = p->d_attn;
    k.hbuf = p->d_h;
    k.rope = p->d_rope;
    k.ctl = p->d_ctl;
    k.cl = p->cl;
    k.tasks = p->d_tasks;
    k.queue_off = p->d_queue;
    for (int i = 0; i < OP_COUNT; ++i) k.mv[i] = g.mv[i];
    k.slot_bytes = g.slot_bytes;
    k.num_slots = g.num_slots;
    k.attn_ts = g.tps;
    k.attn_splits = g.attn_splits;
    k.l2_prefetch_bytes = g.l2_prefetch_bytes;
    k.max_inflight = g.max_inflight;
    k.down_maps = p->d_down_maps;
    k.only_op = -1;
    k.only_layer = -1;
    k.skip_lm = 0;
    k.kv_appended = g.kv_append ? 1 : 0;
    k.jit = g.jit ? 1 : 0;
    k.n_stages = n_stages;
    k.stage_off = p->d_stage_off;
    k.timeout_ns = (uint64_t)p->opt.timeout_ms * 1000000ull;
    k.trace = p->d_trace;
    k.trace_stride = p->trace_stride;
    k.tc = g.tc ? 1 : 0;
    k.num_ctas = g.num_ctas;
    if (g.tc) {
        k.npad = g.npad;
        k.idesc = umma_idesc_bf16(kTcTileM, 2 * g.npad);
        k.h_tiles = g.h_tiles;
        k.aslot_bytes = g.aslot_bytes;
        k.num_aslots = g.num_aslots;
        k.tc_sub = g.tc_sub;
        uint32_t cols = 32;
        while (cols < (uint32_t)(8 * g.npad)) cols <<= 1;  // two buffers x (gate, up) x 2 * npad columns
        k.tmem_cols = cols;
        for (int i = 0; i < OP_COUNT; ++i) k.tcg[i] = g.tcg[i];
        k.tmaps = p->d_tmaps;
        k.xa = p->d_xa;
        k.ssq = p->d_ssq;
        k.attn_a = p->d_attn_a;
        k.h_a = p->d_h_a;
        k.part = p->d_tc_part;
        k.tile_ctr = p->d_ctl + p->cl.tile_idx;
    }
    *out = p;
    return MK_OK;
}

mk_status mk_plan_create(const mk_model_cfg *cfg, const mk_weight_ptrs *w, mk_plan **out) {
    return mk_plan_create_ex(cfg, w, nullptr, out);
}

mk_status mk_decode_step(mk_plan *p, const int32_t *tokens, const int32_t *positions, const mk_kv_cache *kv,
                         float *logits, void *stream) {
    if (!p || !tokens || !positions || !logits) return MK_ERR_INVALID;
    mk_status st = check_kv(p, kv);
    if (st != MK_OK) return st;
    KParams k = step_params(p, tokens, 1, positions, 1, kv, logits);
    return launch_step(p, k, static_cast<cudaStream_t>(stream));
}

mk_status mk_decode_step_greedy(mk_plan *p, int32_t *tokens, int32_t *positions, const mk_kv_cache *kv,
                                float *logits, void *stream) {
    if (!p || !tokens || !positions || !logits) return MK_ERR_INVALID;
    mk_status st = check_kv(p, kv);
    if (st != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    KParams k = step_params(p, tokens, 1, positions, 1, kv, logits);
    k.greedy = 1;
    k.next_tokens = tokens;
    k.next_positions = positions;
    return launch_step(p, k, s);
}

mk_status mk_decode_step_ablation(mk_plan *p, const int32_t *tokens, const int32_t *positions,
                                  const mk_kv_cache *kv, float *logits, void *stream) {
    if (!p || !tokens || !positions || !logits) return MK_ERR_INVALID;
    if (p->tables.g.jit) return MK_ERR_UNSUPPORTED;  // one operator per launch needs the static queues
    mk_status st = check_kv(p, kv);
    if (st != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaSetDevice(p->device) != cudaSuccess) return cuda_status(cudaGetLastError());
    KParams k = step_params(p, tokens, 1, positions, 1, kv, logits);
    if ((st = clear_trace(p, s)) != MK_OK) return st;
    if ((st = poison_scratch(p, s)) != MK_OK) return st;  // once per step: later launches read earlier ones
    static const int kOps[] = {OP_QKV, OP_ATTN, OP_O, OP_GU, OP_DOWN};
    if (p->tables.g.tc) {
        k.only_op = OP_EMBED;
        k.only_layer = 0;
        st = cuda_status(launch_megakernel(k, p->variant, p->tables.g.num_ctas, p->smem, false, s));
        if (st != MK_OK) return st;
    }
    for (int l = 0; l < p->cfg.n_layers; ++l)
        for (int op : kOps) {
            k.only_op = op;
            k.only_layer = l;
            st = cuda_status(launch_megakernel(k, p->variant, p->tables.g.num_ctas, p->smem, false, s));
            if (st != MK_OK) return st;
        }
    k.only_op = OP_LM;
    k.only_layer = p->cfg.n_layers - 1;
    return cuda_status(launch_megakernel(k, p->variant, p->tables.g.num_ctas, p->smem, false, s));
}

}  // extern "C"

namespace {

// Rows of one chunked-prefill launch.
constexpr int32_t kPrefillRows = 64;

// The chunked-prefill engine of a plan: a plan of the same decoder whose
// kPrefillRows batch rows are consecutive tokens of one sequence, run on the
// tensor-core path with the kv-append graph (every row's K/V is in the cache
// before any row attends).  Made on first use.
mk_status ensure_prefill_engine(mk_plan *p) {
    if (p->pre) return MK_OK;
    mk_model_cfg c = p->cfg;
    c.batch = kPrefillRows;
    mk_plan_options o;
    std::memset(&o, 0, sizeof(o));
    o.num_ctas = p->opt.num_ctas;
    o.timeout_ms = p->opt.timeout_ms;
    o.tensor_cores = 1;
    o.kv_append = 1;
    o.test_poison_scratch = p->opt.test_poison_scratch;
    const int L = c.n_layers;
    std::vector<const void *> f[9];
    for (auto &v : f) v.resize(L);
    for (int l = 0; l < L; ++l) {
        const LayerW &w = p->hlw[l];
        const void *ptrs[9] = {w.attn_norm, w.wq, w.wk, w.wv, w.wo, w.mlp_norm, w.w_gate, w.w_up, w.w_down};
        for (int i = 0; i < 9; ++i) f[i][l] = ptrs[i];
    }
    const mk_weight_ptrs w = {p->w_embed, p->w_lm, p->w_final, f[0].data(), f[1].data(), f[2].data(), f[3].data(),
                              f[4].data(), f[5].data(), f[6].data(), f[7].data(), f[8].data()};
    mk_plan *q = nullptr;
    mk_status st = mk_plan_create_ex(&c, &w, &o, &q);
    if (st != MK_OK) return st;
    if ((st = dev_alloc(q, &p->d_pre_logits, (size_t)kPrefillRows * c.vocab)) != MK_OK ||
        (st = dev_alloc(q, &p->d_pre_tok, kPrefillRows)) != MK_OK ||
        (st = dev_alloc(q, &p->d_pre_pos, kPrefillRows)) != MK_OK) {
        free_plan(q);
        return st;
    }
    p->pre = q;
    return MK_OK;
}

// Prefill of the T tokens of batch row `row` (its page-table row) through
// the engine: chunks of up to kPrefillRows consecutive tokens, one launch
// each (the rows past a short last chunk repeat its last token at its
// position: they write the same K/V to the same slot and are not read); the
// LM head runs on the last chunk only, whose last row's logits go to `logits`.
mk_status prefill_seq(mk_plan *p, int32_t row, const int32_t *tokens, int32_t T, const mk_kv_cache *kv,
                      float *logits, cudaStream_t s) {
    mk_plan *q = p->pre;
    mk_status st = check_kv(q, kv);
    if (st != MK_OK) return st;
    const int32_t V = p->cfg.vocab;
    int32_t n = 0;
    for (int32_t c0 = 0; c0 < T; c0 += kPrefillRows) {
        n = std::min(kPrefillRows, T - c0);
        const cudaError_t e = launch_prefill_rows(tokens + c0, n, c0, kPrefillRows, p->d_pre_tok, p->d_pre_pos, s);
        if (e != cudaSuccess) return cuda_status(e);
        KParams k = step_params(q, p->d_pre_tok, 1, p->d_pre_pos, 1, kv, p->d_pre_logits);
        k.page_table = kv->page_table + (int64_t)row * kv->max_pages_per_seq;
        k.pt_stride = 0;  // every row of the launch is a token of this sequence
        k.skip_lm = (c0 + n < T) ? 1 : 0;
        if ((st = launch_step(q, k, s)) != MK_OK) return st;
    }
    return cuda_status(cudaMemcpyAsync(logits, p->d_pre_logits + (int64_t)(n - 1) * V, (size_t)V * sizeof(float),
                                       cudaMemcpyDeviceToDevice, s));
}

}  // namespace

extern "C" {

mk_status mk_prefill(mk_plan *p, const int32_t *tokens, int32_t T, const mk_kv_cache *kv, float *last_logits,
                     void *stream) {
    if (!p || !tokens || !last_logits || T <= 0 || T > p->cfg.max_seq) return MK_ERR_INVALID;
    mk_status st = check_kv(p, kv);
    if (st != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // chunked prefill when a launch of kPrefillRows tokens of one sequence
    // beats a launch of one token of each sequence
    if (T > 1 && p->cfg.batch < kPrefillRows && p->opt.prefill_by_decode == 0 &&
        ensure_prefill_engine(p) == MK_OK) {
        for (int32_t b = 0; b < p->cfg.batch; ++b)
            if ((st = prefill_seq(p, b, tokens + (int64_t)b * T, T, kv, last_logits + (int64_t)b * p->cfg.vocab, s)) !=
                MK_OK)
                return st;
        return MK_OK;
    }
    for (int32_t t = 0; t < T; ++t) {
        KParams k = step_params(p, tokens + t, T, p->d_iota + t, 0, kv, last_logits);
        k.skip_lm = (t + 1 < T) ? 1 : 0;
        if ((st = launch_step(p, k, s)) != MK_OK) return st;
    }
    return MK_OK;
}

mk_status mk_prefill_row(mk_plan *p, int32_t row, const int32_t *tokens, int32_t T, const mk_kv_cache *kv,
                         float *logits, void *stream) {
    if (!p || !tokens || !logits || row < 0 || row >= p->cfg.batch || T <= 0 || T > p->cfg.max_seq)
        return MK_ERR_INVALID;
    mk_status st = check_kv(p, kv);
    if (st != MK_OK) return st;
    if ((st = ensure_prefill_engine(p)) != MK_OK) return st;
    return prefill_seq(p, row, tokens, T, kv, logits, static_cast<cudaStream_t>(stream));
}

mk_status mk_greedy_next(mk_plan *p, const float *logits, int32_t *tokens, int32_t *positions, void *stream) {
    if (!p || !logits || !tokens || !positions) return MK_ERR_INVALID;
    return cuda_status(launch_greedy_next(logits, p->cfg.batch, p->cfg.vocab, tokens, positions,
                                          static_cast<cudaStream_t>(stream)));
}

mk_status mk_plan_last_error(mk_plan *p, void *stream, mk_device_error *info) {
    if (!p) return MK_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // one copy on the plan's stream into pinned memory, then one wait
    cudaError_t e = cudaMemcpyAsync(p->h_err, p->d_ctl + p->cl.err_idx, 4 * sizeof(uint32_t),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    uint32_t words[4];
    std::memcpy(words, p->h_err, sizeof(words));
    if (words[0] != 0) {
        // clear the error, the abort flag and every counter for the next launch
        e = cudaMemsetAsync(p->d_ctl, 0, (size_t)p->cl.total * sizeof(uint32_t), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (info) {
        info->status = (int32_t)words[0];
        info->site = (int32_t)words[1];
        info->cta = (int32_t)words[2];
        info->detail = (int32_t)words[3];
    }
    return (mk_status)words[0];
}

mk_status mk_decode_step_host(mk_plan *p, const int32_t *tokens_host, const int32_t *positions_host,
                              const mk_kv_cache *kv, float *logits_host, void *stream) {
    if (!p || !tokens_host || !positions_host || !logits_host) return MK_ERR_INVALID;
    mk_status st = check_kv(p, kv);
    if (st != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t nb = (size_t)p->cfg.batch * sizeof(int32_t);
    cudaError_t e = cudaMemcpyAsync(p->d_stage_tok, tokens_host, nb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_stage_pos, positions_host, nb, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_status(e);
    KParams k = step_params(p, p->d_stage_tok, 1, p->d_stage_pos, 1, kv, p->d_stage_logits);
    if ((st = launch_step(p, k, s)) != MK_OK) return st;
    e = cudaMemcpyAsync(logits_host, p->d_stage_logits, (size_t)p->cfg.batch * p->cfg.vocab * sizeof(float),
                        cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_status(e);
    return mk_plan_last_error(p, stream, nullptr);
}

mk_status mk_decode_step_greedy_host(mk_plan *p, const int32_t *tokens_host, const int32_t *positions_host,
                                     const mk_kv_cache *kv, int32_t *next_tokens_host, void *stream) {
    if (!p || !tokens_host || !positions_host || !next_tokens_host) return MK_ERR_INVALID;
    mk_status st = check_kv(p, kv);
    if (st != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t nb = (size_t)p->cfg.batch * sizeof(int32_t);
    cudaError_t e = cudaMemcpyAsync(p->d_stage_tok, tokens_host, nb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_stage_pos, positions_host, nb, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_status(e);
    KParams k = step_params(p, p->d_stage_tok, 1, p->d_stage_pos, 1, kv, p->d_stage_logits);
    k.greedy = 1;  // the step rewrites the staged tokens (and positions) with its pick
    k.next_tokens = p->d_stage_tok;
    k.next_positions = p->d_stage_pos;
    if ((st = launch_step(p, k, s)) != MK_OK) return st;
    e = cudaMemcpyAsync(next_tokens_host, p->d_stage_tok, nb, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_status(e);
    return mk_plan_last_error(p, stream, nullptr);
}

mk_status mk_plan_trace(mk_plan *p, void *stream, uint64_t *out, int64_t capacity, int32_t *num_ctas,
                        int32_t *max_tasks) {
    if (!p || !p->d_trace) return MK_ERR_INVALID;
    if (num_ctas) *num_ctas = p->tables.g.num_ctas;
    if (max_tasks) *max_tasks = p->trace_stride;
    const int64_t n = (int64_t)p->tables.g.num_ctas * p->trace_stride * 8;
    if (!out || capacity < n) return MK_ERR_INVALID;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaMemcpy(out, p->d_trace, (size_t)n * sizeof(uint64_t), cudaMemcpyDeviceToHost);
    return cuda_status(e);
}

void mk_plan_destroy(mk_plan *p) {
    if (!p) return;
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    free_plan(p);
}

}  // extern "C"
