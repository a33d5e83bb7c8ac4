// noalloc.cu — a batch-1 decode step that allocates no device memory.
//
// Some callers cannot call cudaMalloc at the time they need a decode step.
// Examples: code that runs while a memory pool or a CUDA graph owns the
// device's allocations, a host runtime that reserves all device memory up
// front, or a process that must not grow its footprint once it is serving.
// mk_decode_step_noalloc serves them. It builds the task graph on the host,
// then runs the same persistent kernel as mk_decode_step. The kernel's
// scratch (task tables, activations, attention partials, RoPE table, event
// counters and error word) lives in one file-scope __device__ array of
// kNoAllocScratchBytes. The caller passes inputs and outputs, as for
// mk_decode_step.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/mk.h"
#include "mk_kernel.h"
#include "planner.h"

using namespace mk;

namespace {

// Fixed scratch of the allocation-free entry point. Every GPU that loads the
// library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// In host code, g_noalloc_scratch names a host-side stand-in, not a device
// address. Its device address is looked up with the device current, once per
// device and CUDA context, and cached here. The context's unique id is kept
// beside it: after cudaDeviceReset the device gets a new primary context, in
// which the array may sit elsewhere, and the address is looked up again.
constexpr int kMaxDevices = 64;
struct ScratchAddr {
    unsigned long long ctx_id = 0;
    void *ptr = nullptr;
};
ScratchAddr g_scratch_dev[kMaxDevices];
std::mutex g_scratch_mu;

// Unique id of the calling thread's current CUDA context (driver entry
// points, looked up once; no libcuda link).
bool current_context_id(unsigned long long *id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    if (!get_current || !get_id) {
        void *f = nullptr, *g = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &g, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return false;
        }
        get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(g);
    }
    CUcontext ctx = nullptr;
    unsigned long long v = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &v) != CUDA_SUCCESS) return false;
    *id = v;
    return true;
}

// Device address of the fixed scratch on `dev`, which must be current.
mk_status scratch_address(int dev, unsigned char **out) {
    if (dev < 0 || dev >= kMaxDevices) return MK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    // makes the device's primary context current (created if need be)
    if (cudaSetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_CUDA;
    }
    unsigned long long id = 0;
    if (!current_context_id(&id)) return MK_ERR_CUDA;
    ScratchAddr &a = g_scratch_dev[dev];
    if (!a.ptr || a.ctx_id != id) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            cudaGetLastError();
            return MK_ERR_CUDA;
        }
        a.ptr = ptr;
        a.ctx_id = id;
    }
    *out = static_cast<unsigned char *>(a.ptr);
    return MK_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bump allocator over the fixed scratch: 256-byte aligned offsets.
struct Carve {
    size_t used = 0;
    size_t take(size_t bytes) {
        const size_t off = (used + 255) / 256 * 256;
        used = off + bytes;
        return off;
    }
};

}  // namespace

extern "C" mk_status mk_decode_step_noalloc(const mk_model_cfg *cfg, const mk_weight_ptrs *w, const int32_t *tokens,
                                            const int32_t *positions, const mk_kv_cache *kv, float *logits,
                                            void *stream) {
    if (!cfg || !w || !tokens || !positions || !kv || !logits) return MK_ERR_INVALID;
    mk_status st = check_cfg(*cfg);
    if (st != MK_OK) return st;
    const mk_model_cfg &c = *cfg;
    if (c.batch != 1) return MK_ERR_UNSUPPORTED;  // the batch-1 matvec path only
    if (!aligned16(w->embed) || !aligned16(w->lm_head) || !aligned16(w->final_norm)) return MK_ERR_INVALID;
    if (c.tied_embeddings && w->lm_head != w->embed) return MK_ERR_INVALID;
    const void *const *arrs[] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->w_gate, w->w_up, w->w_down};
    for (const void *const *a : arrs) {
        if (!a) return MK_ERR_INVALID;
        for (int l = 0; l < c.n_layers; ++l)
            if (!aligned16(a[l])) return MK_ERR_INVALID;
    }
    if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !aligned16(kv->page_table) || kv->num_pages <= 0 ||
        kv->max_pages_per_seq <= 0 || (int64_t)kv->max_pages_per_seq * c.page_size < c.max_seq)
        return MK_ERR_INVALID;

    int dev = 0, sms = 0, smem_optin = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) {
        cudaGetLastError();
        return MK_ERR_CUDA;
    }
    if (!coop) return MK_ERR_UNSUPPORTED;
    unsigned char *scratch = nullptr;
    if ((st = scratch_address(dev, &scratch)) != MK_OK) return st;

    // task graph on the host, default options
    const mk_plan_options opt = resolve_options(c, nullptr, sms);
    PlanTables t;
    if ((st = build_plan(c, opt, &t)) != MK_OK) return st;
    const PlanGeom &g = t.g;

    // carve the fixed scratch
    const int32_t G = c.n_q_heads / c.n_kv_heads, S = g.attn_splits;
    const int32_t qkv_rows = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    const CtlLayout cl = ctl_layout(g.n_events, c.batch * c.n_kv_heads, 0, c.batch);
    Carve cv;
    const size_t o_layers = cv.take(sizeof(LayerW) * c.n_layers);
    const size_t o_tasks = cv.take(sizeof(Task) * t.tasks.size());
    const size_t o_queue = cv.take(sizeof(int32_t) * t.queue_off.size());
    const size_t o_x = cv.take(sizeof(float) * c.hidden);
    const size_t o_qkv = cv.take(sizeof(float) * qkv_rows);
    const size_t o_part = cv.take(sizeof(float) * c.n_kv_heads * S * G * (c.head_dim + 2));
    const size_t o_attn = cv.take(sizeof(float) * c.n_q_heads * c.head_dim);
    const size_t o_h = cv.take(sizeof(float) * c.ffn_dim);
    const size_t o_rope = cv.take(sizeof(float2) * c.max_seq * (c.head_dim / 2));
    const size_t o_ctl = cv.take(sizeof(uint32_t) * cl.total);
    if (cv.used > kNoAllocScratchBytes) return MK_ERR_OOM;  // shape needs more than the fixed scratch

    const size_t smem = megakernel_smem_bytes(g.slot_bytes, g.num_slots, 0, 0);
    if ((int)smem > smem_optin) return MK_ERR_INVALID;
    const int variant = megakernel_variant(std::max({c.hidden, c.ffn_dim, c.n_q_heads * c.head_dim}), false, false);
    int per_sm = 0;
    if (megakernel_set_smem(variant, smem) != cudaSuccess ||
        megakernel_max_active(variant, smem, &per_sm) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_CUDA;
    }
    if (per_sm < 1) return MK_ERR_LAUNCH;

    std::vector<LayerW> lw(c.n_layers);
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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The scratch keeps the previous call's contents: upload this call's
    // tables and clear the control words (counters, abort flag, error word).
    cudaError_t e = cudaMemcpyAsync(scratch + o_layers, lw.data(), lw.size() * sizeof(LayerW),
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(scratch + o_tasks, t.tasks.data(), t.tasks.size() * sizeof(Task), cudaMemcpyHostToDevice,
                            s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(scratch + o_queue, t.queue_off.data(), t.queue_off.size() * sizeof(int32_t),
                            cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch + o_ctl, 0, sizeof(uint32_t) * cl.total, s);
    if (e == cudaSuccess)
        e = launch_rope_table(reinterpret_cast<float2 *>(scratch + o_rope), c.max_seq, c.head_dim, c.rope_theta, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_CUDA;
    }

    KParams k{};
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
    k.layers = reinterpret_cast<const LayerW *>(scratch + o_layers);
    if (!encode_kv_maps(k, c, *kv, g.tps)) return MK_ERR_INVALID;
    k.k_pool = static_cast<uint16_t *>(kv->k_pool);
    k.v_pool = static_cast<uint16_t *>(kv->v_pool);
    k.page_table = kv->page_table;
    k.num_pages = kv->num_pages;
    k.max_pages = kv->max_pages_per_seq;
    k.pt_stride = kv->max_pages_per_seq;
    k.tokens = tokens;
    k.tok_stride = 1;
    k.positions = positions;
    k.pos_stride = 1;
    k.logits = logits;
    k.x = reinterpret_cast<float *>(scratch + o_x);
    k.qkv = reinterpret_cast<float *>(scratch + o_qkv);
    k.attn_part = reinterpret_cast<float *>(scratch + o_part);
    k.attn_out = reinterpret_cast<float *>(scratch + o_attn);
    k.hbuf = reinterpret_cast<float *>(scratch + o_h);
    k.rope = reinterpret_cast<const float2 *>(scratch + o_rope);
    k.ctl = reinterpret_cast<uint32_t *>(scratch + o_ctl);
    k.cl = cl;
    k.tasks = reinterpret_cast<const Task *>(scratch + o_tasks);
    k.queue_off = reinterpret_cast<const int32_t *>(scratch + o_queue);
    for (int i = 0; i < OP_COUNT; ++i) k.mv[i] = g.mv[i];
    k.slot_bytes = g.slot_bytes;
    k.num_slots = g.num_slots;
    k.attn_ts = g.tps;
    k.attn_splits = g.attn_splits;
    k.l2_prefetch_bytes = g.l2_prefetch_bytes;
    k.max_inflight = g.max_inflight;
    k.only_op = -1;
    k.only_layer = -1;
    k.skip_lm = 0;
    k.timeout_ns = (uint64_t)opt.timeout_ms * 1000000ull;
    k.trace = nullptr;
    k.trace_stride = 0;
    k.tc = 0;
    k.num_ctas = g.num_ctas;
    e = launch_megakernel(k, variant, g.num_ctas, smem, true, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorCooperativeLaunchTooLarge ? MK_ERR_LAUNCH : MK_ERR_CUDA;
    }
    // device-detected errors (bounds, timeouts) come back through the error word
    uint32_t words[4] = {0, 0, 0, 0};
    e = cudaMemcpyAsync(words, scratch + o_ctl + sizeof(uint32_t) * cl.err_idx, sizeof(words), cudaMemcpyDeviceToHost,
                        s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_CUDA;
    }
    return (mk_status)words[0];
}
