// megakernel.cu — the persistent decode megakernel for B300 (sm_103a).
//
// One cooperative launch runs one decode step.  Every SM hosts one worker CTA
// (the MPK runtime's "worker" with a dedicated task queue, "Compilar LLM en un
// MegaKernel…", section "Parte 2. Runtime / Workers") made of three roles:
//
//  * warp 0 — scheduler: walks the CTA's queue and, for each task, spins on
//    the global event counter the task depends on (a counter with a
//    threshold, section "Método de ejecución basado en eventos"), then hands
//    the task to the compute warps through shared memory.  One scheduler
//    warp per SM, as in section "Schedulers".
//  * warp 1 — producer: walks the same queue AHEAD of the compute warps and
//    streams every task's immutable operands (weight rows, past KV entries)
//    into a ring of shared-memory slots with bulk async copies completed on
//    mbarriers.  Weights never depend on activations, so the stream crosses
//    task and layer boundaries: the next task's data is loading while the
//    current task computes, which is the paged shared memory of "MPK: A
//    Compiler and Runtime for Mega-Kernelizing Tensor Programs" (section 4)
//    and the cross-layer software pipelining of "Compilar LLM…", section
//    "Panorama general".
//  * warps 2..9 — compute: run the fused task bodies (RMSNorm + QKV; RoPE +
//    KV append + split attention; split merge + O-proj + residual; RMSNorm +
//    gate/up + SiLU*mul; down + residual; final RMSNorm + LM head — the fused
//    instruction list of "Llama-70B 向け…megakernel", section
//    高スループットMegakernelの設計と工夫) and signal the task's event
//    with a gpu-scope release.
//
// Matrix-vector tasks: each compute thread owns fixed 16-byte column chunks
// of the input vector and keeps them (normalised) in registers for the whole
// task; weight rows are read from the ring once with 128-bit shared loads;
// per-row sums are reduced with warp shuffles and one cross-warp step.
//
// Every wait is bounded by the plan's time budget; on expiry the kernel
// records an error, raises a grid-wide abort flag, drains its own copies in
// flight and returns.  Compute warps never leave a sequence of named
// barriers early: a failed wait only marks the CTA aborted, and all compute
// warps stop together at the next task boundary.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mk_kernel.h"
#include "ptx.cuh"

namespace mk {

namespace {

struct SmemCtl {
    uint64_t full[kMaxSlots];
    uint64_t empty[kMaxSlots];
    uint32_t ready;      // tasks [0, ready) of the queue have their dependencies met
    uint32_t abort;      // local abort flag
    uint32_t last_flag;  // attention: this CTA finished the last split of a head
    uint32_t pad0;
    float red[2][kComputeWarps][8];
    float rms_part[kComputeWarps];
    float att_m[kMaxGroup], att_l[kMaxGroup], att_alpha[kMaxGroup];
    alignas(16) float q_s[kMaxGroup][kMaxHeadDim];
    alignas(16) float s_s[kMaxGroup][kMaxTps];
    alignas(16) uint16_t knew[kMaxHeadDim];
    alignas(16) uint16_t vnew[kMaxHeadDim];
};

constexpr size_t kRingOffset = (sizeof(SmemCtl) + 1023) / 1024 * 1024;
constexpr uint32_t kReadyAbort = 0x7FFFFFFFu;

struct Ctx {
    const KParams *p;
    SmemCtl *sc;
    uint8_t *ring;
    int cta;
};

__device__ __forceinline__ bool task_active(const KParams &p, const Task &t) {
    if (p.only_op >= 0) return t.op == p.only_op && t.layer == p.only_layer;
    if (p.skip_lm && t.op == OP_LM) return false;
    return true;
}

__device__ __forceinline__ uint64_t *trace_slot(const KParams &p, int task) {
    return p.trace ? p.trace + ((size_t)blockIdx.x * p.trace_stride + task) * 8 : nullptr;
}

__device__ __forceinline__ bool global_abort(const KParams &p) {
    return ld_relaxed_gpu(p.ctl + p.cl.abort_idx) != 0;
}

__device__ __forceinline__ bool local_abort(const Ctx &c) { return *(volatile uint32_t *)&c.sc->abort != 0; }
__device__ __forceinline__ void set_local_abort(const Ctx &c) { *(volatile uint32_t *)&c.sc->abort = 1u; }

__device__ void record_error(const Ctx &c, int32_t status, int32_t site, int32_t detail) {
    const KParams &p = *c.p;
    uint32_t *err = p.ctl + p.cl.err_idx;
    if (atomicCAS(err, 0u, (uint32_t)status) == 0u) {
        volatile uint32_t *e = err;
        e[1] = (uint32_t)site;
        e[2] = (uint32_t)c.cta;
        e[3] = (uint32_t)detail;
    }
    __threadfence();
    atomicExch(p.ctl + p.cl.abort_idx, 1u);
    set_local_abort(c);
}

// Bounded wait on an mbarrier phase.  Returns false on abort or timeout; a
// failure always leaves the CTA marked aborted.
__device__ bool wait_mbar(const Ctx &c, uint64_t *bar, uint32_t parity, int32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (local_abort(c) || global_abort(*c.p)) {
                set_local_abort(c);
                return false;
            }
            if (globaltimer_ns() - t0 > c.p->timeout_ns) {
                record_error(c, 4 /*MK_ERR_TIMEOUT*/, site, (int32_t)parity);
                return false;
            }
        }
    }
}

// ----------------------------------------------------------------- pages
// A task's immutable operands are cut into ring-slot "pages"; producer and
// consumers enumerate them with the same loops.

__device__ __forceinline__ int32_t qkv_boundary(const KParams &p, int32_t row) {
    const int32_t qr = p.nq * p.d, kr = qr + p.nkv * p.d;
    return row < qr ? qr : (row < kr ? kr : p.qkv_rows);
}

__device__ __forceinline__ int32_t mv_group_rows(const KParams &p, int op, int32_t row, int32_t row_end) {
    int32_t n = min(p.mv[op].rpp, row_end - row);
    if (op == OP_QKV) n = min(n, qkv_boundary(p, row) - row);
    return n;
}

// matrix and local row of operator row `row`
__device__ __forceinline__ const uint16_t *mv_matrix(const KParams &p, int op, int layer, int32_t row,
                                                     int32_t *local) {
    const LayerW &w = p.layers[layer];
    *local = row;
    switch (op) {
        case OP_QKV: {
            const int32_t qr = p.nq * p.d, kr = qr + p.nkv * p.d;
            if (row < qr) return w.wq;
            if (row < kr) {
                *local = row - qr;
                return w.wk;
            }
            *local = row - kr;
            return w.wv;
        }
        case OP_O: return w.wo;
        case OP_GU: return w.w_gate;
        case OP_DOWN: return w.w_down;
        default: return p.lm_head;
    }
}

struct AttnRange {
    int32_t pos, lo, cend;  // cached tokens [lo, cend); new token at pos
    bool has_new;
};

// Split s of S covers context positions [s*C/S, (s+1)*C/S) of C = pos + 1;
// the last split always holds the new token.
__device__ __forceinline__ AttnRange attn_range(const KParams &p, const Task &t) {
    AttnRange r;
    r.pos = p.positions[(int64_t)t.a0 * p.pos_stride];
    const int64_t C = (int64_t)r.pos + 1;
    r.lo = (int32_t)((int64_t)t.a2 * C / t.a3);
    const int32_t hi = (int32_t)((int64_t)(t.a2 + 1) * C / t.a3);
    r.cend = min(hi, r.pos);
    r.has_new = (t.a2 == t.a3 - 1);
    return r;
}

__device__ __forceinline__ int64_t kv_offset(const KParams &p, int layer, int32_t page, int32_t kvh, int32_t slot) {
    return (((int64_t)layer * p.num_pages + page) * p.nkv + kvh) * (int64_t)p.page_size * p.d + (int64_t)slot * p.d;
}

// ------------------------------------------------------------- producer

struct Producer {
    uint32_t issued = 0;
    uint64_t pol;
    uint64_t *tr = nullptr;  // trace entry of the current task

    __device__ bool acquire_slot(const Ctx &c, uint32_t *slot) {
        const uint32_t s = issued % (uint32_t)c.p->num_slots;
        const uint32_t round = issued / (uint32_t)c.p->num_slots;
        const uint64_t t0 = tr ? globaltimer_ns() : 0;
        if (!wait_mbar(c, &c.sc->empty[s], (round & 1u) ^ 1u, SITE_EMPTY_WAIT)) return false;
        if (tr) {
            const uint64_t t1 = globaltimer_ns();
            if (tr[4] == 0) tr[4] = t1;
            tr[5] += t1 - t0;
        }
        *slot = s;
        return true;
    }

    __device__ bool run_matvec(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const int op = t.op;
        const MvGeom &g = p.mv[op];
        for (int32_t row = t.a0; row < t.a1;) {
            const int32_t n = mv_group_rows(p, op, row, t.a1);
            int32_t lr;
            const uint16_t *W = mv_matrix(p, op, t.layer, row, &lr);
            for (int32_t ks = 0; ks < g.ksplit; ++ks) {
                uint32_t s;
                if (!acquire_slot(c, &s)) return false;
                const int32_t k0 = ks * g.kc;
                const int32_t pw = min(g.kc, g.K - k0);
                const uint32_t bytes = (uint32_t)(g.row_mult * n * pw * 2);
                uint8_t *dst = c.ring + (size_t)s * p.slot_bytes;
                mbar_arrive_expect_tx(&c.sc->full[s], bytes);
                for (int m = 0; m < g.row_mult; ++m) {
                    const uint16_t *Wm = (m == 0) ? W : p.layers[t.layer].w_up;
                    if (g.ksplit == 1) {
                        bulk_g2s(dst + (size_t)m * n * pw * 2, Wm + (int64_t)lr * g.K, (uint32_t)(n * pw * 2),
                                 &c.sc->full[s], pol);
                    } else {
                        for (int32_t r = 0; r < n; ++r)
                            bulk_g2s(dst + (size_t)(m * n + r) * pw * 2, Wm + (int64_t)(lr + r) * g.K + k0,
                                     (uint32_t)(pw * 2), &c.sc->full[s], pol);
                    }
                }
                ++issued;
            }
            row += n;
        }
        return true;
    }

    __device__ bool run_attn(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const AttnRange r = attn_range(p, t);
        const int32_t tps = p.tps;
        const int32_t *pt = p.page_table + (int64_t)t.a0 * p.max_pages;
        for (int32_t t0 = r.lo; t0 < r.cend; t0 += tps) {
            const int32_t t1 = min(r.cend, t0 + tps);
            uint32_t s;
            if (!acquire_slot(c, &s)) return false;
            uint8_t *dst = c.ring + (size_t)s * p.slot_bytes;
            mbar_arrive_expect_tx(&c.sc->full[s], (uint32_t)(2 * (t1 - t0) * p.d * 2));
            for (int32_t tt = t0; tt < t1;) {
                const int32_t pg = pt[tt / p.page_size];
                const int32_t n = min(t1, (tt / p.page_size + 1) * p.page_size) - tt;
                const int64_t off = kv_offset(p, t.layer, pg, t.a1, tt % p.page_size);
                const uint32_t bytes = (uint32_t)(n * p.d * 2);
                bulk_g2s(dst + (size_t)(tt - t0) * p.d * 2, p.k_pool + off, bytes, &c.sc->full[s], pol);
                bulk_g2s(dst + ((size_t)tps + (tt - t0)) * p.d * 2, p.v_pool + off, bytes, &c.sc->full[s], pol);
                tt += n;
            }
            ++issued;
        }
        return true;
    }

    // Wait for the copies of every slot's most recent page (abort path and
    // normal exit alike), so that no copy is in flight when the CTA exits.
    __device__ void drain(const Ctx &c) {
        const uint32_t ns = (uint32_t)c.p->num_slots;
        const uint32_t lim = issued < ns ? issued : ns;
        for (uint32_t s = 0; s < lim; ++s) {
            const uint32_t k = issued - 1 - ((issued - 1 - s) % ns);  // last page issued on slot s
            const uint32_t par = (k / ns) & 1u;
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&c.sc->full[s], par)) {
                if (globaltimer_ns() - t0 > c.p->timeout_ns) {
                    record_error(c, 4, SITE_DRAIN_WAIT, (int32_t)s);
                    break;
                }
            }
        }
    }
};

__device__ void producer_role(const Ctx &c, const Task *q, int nt) {
    if ((threadIdx.x & 31) != 0) return;
    Producer pr;
    pr.pol = policy_evict_first();
    for (int i = 0; i < nt; ++i) {
        const Task t = q[i];
        if (!task_active(*c.p, t)) continue;
        pr.tr = trace_slot(*c.p, i);
        const bool ok = (t.op == OP_ATTN) ? pr.run_attn(c, t) : pr.run_matvec(c, t);
        if (!ok) break;
    }
    pr.drain(c);
}

// ------------------------------------------------------------ scheduler

__device__ void scheduler_role(const Ctx &c, const Task *q, int nt) {
    if ((threadIdx.x & 31) != 0) return;
    const KParams &p = *c.p;
    const bool use_events = p.only_op < 0;
    for (int i = 0; i < nt; ++i) {
        const Task t = q[i];
        if (use_events && task_active(p, t) && t.wait_ev != kNoEvent) {
            const uint32_t *ctr = p.ctl + t.wait_ev;
            if (ld_acquire_gpu(ctr) < t.wait_count) {
                uint64_t t0 = globaltimer_ns();
                for (uint32_t it = 1;; ++it) {
                    if (ld_acquire_gpu(ctr) >= t.wait_count) break;
                    if ((it & 7u) == 0) {
                        if (local_abort(c) || global_abort(p)) {
                            set_local_abort(c);
                            st_release_cta(&c.sc->ready, kReadyAbort);
                            return;
                        }
                        if (globaltimer_ns() - t0 > p.timeout_ns) {
                            record_error(c, 4, SITE_EVENT_WAIT, t.wait_ev);
                            st_release_cta(&c.sc->ready, kReadyAbort);
                            return;
                        }
                    }
                }
            }
        }
        if (uint64_t *tr = trace_slot(p, i)) tr[0] = globaltimer_ns();
        st_release_cta(&c.sc->ready, (uint32_t)(i + 1));
    }
}

// --------------------------------------------------------- compute warps

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ void compute_bar() { named_bar_sync(1, kComputeThreads); }

__device__ __forceinline__ float dot8(const uint4 w, const float *x) {
    float a = bf16_lo(w.x) * x[0];
    a = fmaf(bf16_hi(w.x), x[1], a);
    a = fmaf(bf16_lo(w.y), x[2], a);
    a = fmaf(bf16_hi(w.y), x[3], a);
    a = fmaf(bf16_lo(w.z), x[4], a);
    a = fmaf(bf16_hi(w.z), x[5], a);
    a = fmaf(bf16_lo(w.w), x[6], a);
    a = fmaf(bf16_hi(w.w), x[7], a);
    return a;
}

struct Consumer {
    uint32_t consumed = 0;
    int ct, wc, lane;  // compute-thread index, compute-warp index, lane
    uint32_t red_buf = 0;
    bool tracing = false;
    uint64_t full_wait_ns = 0;

    // A failed wait (abort or timeout) marks the CTA aborted but keeps the
    // control flow: all compute warps must reach the same named barriers, so
    // they leave only together, at a task boundary.
    __device__ uint32_t wait_slot(const Ctx &c) {
        const uint32_t s = consumed % (uint32_t)c.p->num_slots;
        const uint32_t round = consumed / (uint32_t)c.p->num_slots;
        const uint64_t t0 = tracing ? globaltimer_ns() : 0;
        wait_mbar(c, &c.sc->full[s], round & 1u, SITE_FULL_WAIT);
        if (tracing) full_wait_ns += globaltimer_ns() - t0;
        return s;
    }

    __device__ void release_slot(const Ctx &c, uint32_t s) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.sc->empty[s]);
        ++consumed;
    }

    // ------------------------------------------------------- matvec task
    template <int MAXCH>
    __device__ void run_matvec(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const int op = t.op;
        const MvGeom &g = p.mv[op];
        const int32_t nchunk = g.K / 8;
        const LayerW &lw = p.layers[t.layer];
        const int32_t token = p.tokens[0];

        // input vector for this thread's chunks c = ct + 256 j
        float xr[MAXCH][8];
        const bool from_embed = (op == OP_QKV && t.layer == 0);
        const float *xin = (op == OP_O) ? p.attn_out : (op == OP_DOWN ? p.hbuf : p.x);
        const uint16_t *gain =
            op == OP_QKV ? lw.attn_norm : (op == OP_GU ? lw.mlp_norm : (op == OP_LM ? p.final_norm : nullptr));
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < MAXCH; ++j) {
            const int32_t ch = ct + kComputeThreads * j;
            if (ch < nchunk) {
                if (from_embed) {
                    const uint4 e = __ldg(reinterpret_cast<const uint4 *>(p.embed + (int64_t)token * p.H) + ch);
                    xr[j][0] = bf16_lo(e.x); xr[j][1] = bf16_hi(e.x);
                    xr[j][2] = bf16_lo(e.y); xr[j][3] = bf16_hi(e.y);
                    xr[j][4] = bf16_lo(e.z); xr[j][5] = bf16_hi(e.z);
                    xr[j][6] = bf16_lo(e.w); xr[j][7] = bf16_hi(e.w);
                } else {
                    const float4 a = ld_cg_f4(xin + ch * 8), b = ld_cg_f4(xin + ch * 8 + 4);
                    xr[j][0] = a.x; xr[j][1] = a.y; xr[j][2] = a.z; xr[j][3] = a.w;
                    xr[j][4] = b.x; xr[j][5] = b.y; xr[j][6] = b.z; xr[j][7] = b.w;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(xr[j][e], xr[j][e], ss);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xr[j][e] = 0.f;
            }
        }
        if (gain != nullptr) {
            // RMSNorm: r = 1/sqrt(mean(x^2) + eps), x-hat = g * x * r
            ss = warp_sum(ss);
            if (lane == 0) c.sc->rms_part[wc] = ss;
            compute_bar();
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kComputeWarps; ++w) tot += c.sc->rms_part[w];
            const float r = rsqrtf(tot / (float)g.K + p.eps);
            compute_bar();  // rms_part is reused by the next task
#pragma unroll
            for (int j = 0; j < MAXCH; ++j) {
                const int32_t ch = ct + kComputeThreads * j;
                if (ch < nchunk) {
                    const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(gain) + ch);
                    xr[j][0] *= r * bf16_lo(gv.x); xr[j][1] *= r * bf16_hi(gv.x);
                    xr[j][2] *= r * bf16_lo(gv.y); xr[j][3] *= r * bf16_hi(gv.y);
                    xr[j][4] *= r * bf16_lo(gv.z); xr[j][5] *= r * bf16_hi(gv.z);
                    xr[j][6] *= r * bf16_lo(gv.w); xr[j][7] *= r * bf16_hi(gv.w);
                }
            }
        }

        for (int32_t row = t.a0; row < t.a1;) {
            const int32_t n = mv_group_rows(p, op, row, t.a1);
            const int32_t R = n * g.row_mult;
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = 0.f;
            for (int32_t ks = 0; ks < g.ksplit; ++ks) {
                const uint32_t s = wait_slot(c);
                const int32_t c_lo = ks * (g.kc / 8);
                const int32_t pw8 = min(g.kc / 8, nchunk - c_lo);  // chunks in this piece
                const uint4 *base = reinterpret_cast<const uint4 *>(c.ring + (size_t)s * p.slot_bytes);
#pragma unroll
                for (int j = 0; j < MAXCH; ++j) {
                    const int32_t cl = ct + kComputeThreads * j - c_lo;
                    if (cl >= 0 && cl < pw8) {
#pragma unroll
                        for (int r = 0; r < 8; ++r) {
                            if (r < R) acc[r] += dot8(base[r * pw8 + cl], xr[j]);
                        }
                    }
                }
                release_slot(c, s);
            }
            // reduce the R row sums over the 256 compute threads
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if (r < R) {
                    const float v = warp_sum(acc[r]);
                    if (lane == 0) c.sc->red[red_buf][wc][r] = v;
                }
            }
            compute_bar();
            if (ct < n) {
                float tot = 0.f, tot2 = 0.f;
#pragma unroll
                for (int w = 0; w < kComputeWarps; ++w) tot += c.sc->red[red_buf][w][ct];
                if (g.row_mult == 2) {
#pragma unroll
                    for (int w = 0; w < kComputeWarps; ++w) tot2 += c.sc->red[red_buf][w][n + ct];
                }
                const int32_t orow = row + ct;
                switch (op) {
                    case OP_QKV: p.qkv[orow] = tot; break;
                    case OP_O: {
                        const float xo = (t.layer == 0)
                                             ? __uint_as_float((uint32_t)p.embed[(int64_t)token * p.H + orow] << 16)
                                             : __ldcg(p.x + orow);
                        p.x[orow] = xo + tot;
                        break;
                    }
                    case OP_GU: p.hbuf[orow] = tot / (1.f + expf(-tot)) * tot2; break;
                    case OP_DOWN: p.x[orow] = __ldcg(p.x + orow) + tot; break;
                    default: p.logits[orow] = tot; break;
                }
            }
            red_buf ^= 1u;
            row += n;
        }
    }

    // ---------------------------------------------------- attention task
    // Scores, online-softmax update and value accumulation for ntok tokens
    // whose K rows start at kp and V rows at vp (bf16 [ntok][d] in smem).
    __device__ void attn_block(const Ctx &c, const uint16_t *kp, const uint16_t *vp, int32_t ntok, int G,
                               float *o_acc, int npairs_mine) {
        const KParams &p = *c.p;
        const int d = p.d;
        const int nck = d / 64;  // 16-byte chunks per lane
        const int t_sub = lane >> 3, part = lane & 7;
        SmemCtl *sc = c.sc;
        // scores: 4 tokens per warp per pass, 8 lanes per token
        for (int32_t base = 0; base < ntok; base += kComputeWarps * 4) {
            const int32_t tok = base + wc * 4 + t_sub;
            const bool valid = tok < ntok;
            float acc[kMaxGroup];
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g) acc[g] = 0.f;
            if (valid) {
                for (int i = 0; i < nck; ++i) {
                    const int chunk = part + 8 * ((i + t_sub) % nck);
                    const uint4 kv = reinterpret_cast<const uint4 *>(kp + (size_t)tok * d)[chunk];
                    const float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                                         bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
                    for (int g = 0; g < kMaxGroup; ++g) {
                        if (g < G) {
                            const float4 qa = *reinterpret_cast<const float4 *>(&sc->q_s[g][chunk * 8]);
                            const float4 qb = *reinterpret_cast<const float4 *>(&sc->q_s[g][chunk * 8 + 4]);
                            float a = acc[g];
                            a = fmaf(kf[0], qa.x, a); a = fmaf(kf[1], qa.y, a);
                            a = fmaf(kf[2], qa.z, a); a = fmaf(kf[3], qa.w, a);
                            a = fmaf(kf[4], qb.x, a); a = fmaf(kf[5], qb.y, a);
                            a = fmaf(kf[6], qb.z, a); a = fmaf(kf[7], qb.w, a);
                            acc[g] = a;
                        }
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g) {
                float v = acc[g];
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
                if (g < G && valid && part == 0) sc->s_s[g][tok] = v;
            }
        }
        compute_bar();
        // online softmax: warp g owns head g
        if (wc < G) {
            const int g = wc;
            float mx = -INFINITY;
            for (int32_t tk = lane; tk < ntok; tk += 32) mx = fmaxf(mx, sc->s_s[g][tk]);
            mx = warp_max(mx);
            const float m_old = sc->att_m[g];
            const float m_new = fmaxf(m_old, mx);
            float sum = 0.f;
            for (int32_t tk = lane; tk < ntok; tk += 32) {
                const float e = expf(sc->s_s[g][tk] - m_new);
                sc->s_s[g][tk] = e;
                sum += e;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                const float alpha = expf(m_old - m_new);  // 0 when m_old = -inf
                sc->att_alpha[g] = alpha;
                sc->att_l[g] = sc->att_l[g] * alpha + sum;
                sc->att_m[g] = m_new;
            }
        }
        compute_bar();
        // o = o * alpha + sum_t p_t v_t; this thread owns pairs ct + 256 k
        const int half = d / 2;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (k < npairs_mine) {
                const int pr = ct + kComputeThreads * k;
                const int g = pr / half, e = (pr % half) * 2;
                float o0 = o_acc[2 * k] * sc->att_alpha[g], o1 = o_acc[2 * k + 1] * sc->att_alpha[g];
                for (int32_t tk = 0; tk < ntok; ++tk) {
                    const uint32_t v2 = *reinterpret_cast<const uint32_t *>(vp + (size_t)tk * d + e);
                    const float pw = sc->s_s[g][tk];
                    o0 = fmaf(pw, bf16_lo(v2), o0);
                    o1 = fmaf(pw, bf16_hi(v2), o1);
                }
                o_acc[2 * k] = o0;
                o_acc[2 * k + 1] = o1;
            }
        }
    }

    __device__ void run_attn(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        SmemCtl *sc = c.sc;
        const int d = p.d, half = d / 2;
        const int G = p.nq / p.nkv;
        const int b = t.a0, kvh = t.a1, S = t.a3;
        const AttnRange r = attn_range(p, t);
        const float *qkv = p.qkv + (int64_t)b * p.qkv_rows;
        const float2 *rope = p.rope + (int64_t)r.pos * half;
        const float scale = rsqrtf((float)d);

        // RoPE'd, pre-scaled queries of the G heads sharing this kv head
        for (int idx = ct; idx < G * half; idx += kComputeThreads) {
            const int g = idx / half, i = idx % half;
            const float *qh = qkv + (int64_t)(kvh * G + g) * d;
            const float a = __ldcg(qh + i), bb = __ldcg(qh + i + half);
            const float2 cs = rope[i];
            sc->q_s[g][i] = (a * cs.x - bb * cs.y) * scale;
            sc->q_s[g][i + half] = (a * cs.y + bb * cs.x) * scale;
        }
        if (r.has_new) {
            // K/V of the new token: RoPE on k, round to bf16, append to the cache
            const float *kh = qkv + (int64_t)p.nq * d + (int64_t)kvh * d;
            const float *vh = qkv + (int64_t)(p.nq + p.nkv) * d + (int64_t)kvh * d;
            const int32_t pg = p.page_table[(int64_t)b * p.max_pages + r.pos / p.page_size];
            const int64_t off = kv_offset(p, t.layer, pg, kvh, r.pos % p.page_size);
            for (int i = ct; i < half; i += kComputeThreads) {
                const float a = __ldcg(kh + i), bb = __ldcg(kh + i + half);
                const float2 cs = rope[i];
                const uint16_t k0 = f32_to_bf16_bits(a * cs.x - bb * cs.y);
                const uint16_t k1 = f32_to_bf16_bits(a * cs.y + bb * cs.x);
                sc->knew[i] = k0;
                sc->knew[i + half] = k1;
                p.k_pool[off + i] = k0;
                p.k_pool[off + i + half] = k1;
            }
            for (int i = ct; i < d; i += kComputeThreads) {
                const uint16_t v = f32_to_bf16_bits(__ldcg(vh + i));
                sc->vnew[i] = v;
                p.v_pool[off + i] = v;
            }
        }
        if (ct < G) {
            sc->att_m[ct] = -INFINITY;
            sc->att_l[ct] = 0.f;
        }
        compute_bar();

        const int npairs = G * half;
        const int mine = (ct < npairs) ? (npairs - ct + kComputeThreads - 1) / kComputeThreads : 0;
        float o_acc[4] = {0.f, 0.f, 0.f, 0.f};  // up to 2 pairs per thread (G*d/2 <= 512)
        for (int32_t t0 = r.lo; t0 < r.cend; t0 += p.tps) {
            const int32_t ntok = min(r.cend, t0 + p.tps) - t0;
            const uint32_t s = wait_slot(c);
            const uint16_t *kp = reinterpret_cast<const uint16_t *>(c.ring + (size_t)s * p.slot_bytes);
            attn_block(c, kp, kp + (size_t)p.tps * d, ntok, G, o_acc, mine);
            release_slot(c, s);
            compute_bar();  // scores buffer reused by the next block
        }
        if (r.has_new) {
            attn_block(c, sc->knew, sc->vnew, 1, G, o_acc, mine);
            compute_bar();
        }
        // partial result of this split: unnormalised o, running max, sum
        const int64_t pidx = (((int64_t)b * p.nkv + kvh) * S + t.a2) * G;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (k < mine) {
                const int pr = ct + kComputeThreads * k;
                const int g = pr / half, e = (pr % half) * 2;
                float *dst = p.attn_part + (pidx + g) * (d + 2);
                dst[e] = o_acc[2 * k];
                dst[e + 1] = o_acc[2 * k + 1];
            }
        }
        if (ct < G) {
            float *dst = p.attn_part + (pidx + ct) * (d + 2);
            dst[d] = sc->att_m[ct];
            dst[d + 1] = sc->att_l[ct];
        }
        compute_bar();
        uint32_t *done = p.ctl + p.cl.n_events + b * p.nkv + kvh;
        if (ct == 0) {
            __threadfence();
            const uint32_t old = atom_acq_rel_gpu_add(done, 1u);
            sc->last_flag = (old == (uint32_t)(S - 1)) ? 1u : 0u;
        }
        compute_bar();
        if (sc->last_flag) {
            // last split of this (sequence, kv head): merge the S partials
            if (ct == 0) *done = 0u;  // nothing else touches it in this launch
            const int64_t pbase = ((int64_t)b * p.nkv + kvh) * S * G;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (k < mine) {
                    const int pr = ct + kComputeThreads * k;
                    const int g = pr / half, e = (pr % half) * 2;
                    float M = -INFINITY;
                    for (int s = 0; s < S; ++s)
                        M = fmaxf(M, __ldcg(p.attn_part + (pbase + (int64_t)s * G + g) * (d + 2) + d));
                    float Ls = 0.f, o0 = 0.f, o1 = 0.f;
                    for (int s = 0; s < S; ++s) {
                        const float *src = p.attn_part + (pbase + (int64_t)s * G + g) * (d + 2);
                        const float ms = __ldcg(src + d);
                        const float w = (ms == -INFINITY) ? 0.f : expf(ms - M);
                        Ls = fmaf(__ldcg(src + d + 1), w, Ls);
                        o0 = fmaf(__ldcg(src + e), w, o0);
                        o1 = fmaf(__ldcg(src + e + 1), w, o1);
                    }
                    float *dst = p.attn_out + (int64_t)b * p.nq * d + (int64_t)(kvh * G + g) * d;
                    dst[e] = o0 / Ls;
                    dst[e + 1] = o1 / Ls;
                }
            }
            compute_bar();
            if (ct == 0 && p.only_op < 0 && t.signal_ev != kNoEvent && !local_abort(c)) {
                __threadfence();
                red_release_gpu_add(p.ctl + t.signal_ev, 1u);
            }
        }
    }
};

template <int MAXCH>
__device__ void compute_role(const Ctx &c, const Task *q, int nt) {
    const KParams &p = *c.p;
    Consumer cs;
    cs.ct = threadIdx.x - 64;
    cs.wc = cs.ct >> 5;
    cs.lane = threadIdx.x & 31;
    cs.tracing = p.trace != nullptr && cs.ct == 0;
    for (int i = 0; i < nt; ++i) {
        const Task t = q[i];
        if (!task_active(p, t)) continue;
        // wait for the scheduler to release task i
        if (ld_acquire_cta(&c.sc->ready) < (uint32_t)(i + 1)) {
            uint64_t t0 = globaltimer_ns();
            for (uint32_t it = 1;; ++it) {
                if (ld_acquire_cta(&c.sc->ready) >= (uint32_t)(i + 1)) break;
                if ((it & 63u) == 0) {
                    if (local_abort(c)) break;
                    if (globaltimer_ns() - t0 > 4 * p.timeout_ns) {
                        record_error(c, 4, SITE_READY_WAIT, i);
                        break;
                    }
                }
            }
        }
        compute_bar();  // every compute warp sees the same abort state
        if (local_abort(c)) return;
        uint64_t *tr = cs.tracing ? trace_slot(p, i) : nullptr;
        if (tr) tr[1] = globaltimer_ns();
        if (t.op == OP_ATTN) cs.run_attn(c, t);
        else cs.run_matvec<MAXCH>(c, t);
        compute_bar();  // every output row of the task is written
        if (tr) {
            tr[2] = globaltimer_ns();
            tr[3] = cs.full_wait_ns;
            cs.full_wait_ns = 0;
        }
        if (local_abort(c)) return;
        if (t.op != OP_ATTN && p.only_op < 0 && t.signal_ev != kNoEvent && cs.ct == 0) {
            __threadfence();
            red_release_gpu_add(p.ctl + t.signal_ev, 1u);
        }
    }
}

template <int MAXCH>
__global__ void __launch_bounds__(kThreads, 1) megakernel(const __grid_constant__ KParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SmemCtl *sc = reinterpret_cast<SmemCtl *>(smem_raw);
    Ctx c{&p, sc, smem_raw + kRingOffset, (int)blockIdx.x};
    const Task *q = p.tasks + p.queue_off[blockIdx.x];
    const int nt = p.queue_off[blockIdx.x + 1] - p.queue_off[blockIdx.x];
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.num_slots; ++s) {
            mbar_init(&sc->full[s], 1);
            mbar_init(&sc->empty[s], kComputeWarps);
        }
        sc->ready = 0;
        sc->abort = global_abort(p) ? 1u : 0u;  // a recorded error stays sticky
        sc->last_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // validate this step's inputs before any address is formed from them
    if (threadIdx.x < 32 && !sc->abort) {
        for (int b = threadIdx.x; b < p.B; b += 32) {
            const int32_t tok = p.tokens[(int64_t)b * p.tok_stride];
            const int32_t pos = p.positions[(int64_t)b * p.pos_stride];
            if (tok < 0 || tok >= p.V) {
                record_error(c, 5 /*MK_ERR_BOUNDS*/, SITE_TOKEN, tok);
                continue;
            }
            if (pos < 0 || pos >= p.max_seq || pos / p.page_size >= p.max_pages) {
                record_error(c, 5, SITE_POSITION, pos);
                continue;
            }
            for (int32_t j = 0; j <= pos / p.page_size; ++j) {
                const int32_t pg = p.page_table[(int64_t)b * p.max_pages + j];
                if (pg < 0 || pg >= p.num_pages) {
                    record_error(c, 5, SITE_PAGE, pg);
                    break;
                }
            }
        }
    }
    __syncthreads();
    if (!local_abort(c)) {
        if (warp == kWarpSched) scheduler_role(c, q, nt);
        else if (warp == kWarpProd) producer_role(c, q, nt);
        else compute_role<MAXCH>(c, q, nt);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // the last CTA out resets the counters for the next launch
        __threadfence();
        uint32_t *ex = p.ctl + p.cl.exit_idx;
        const uint32_t old = atom_acq_rel_gpu_add(ex, 1u);
        if (old == gridDim.x - 1) {
            for (int i = 0; i < p.cl.n_events + p.cl.n_done; ++i) p.ctl[i] = 0u;
            *ex = 0u;
            __threadfence();
        }
    }
}

__global__ void rope_table_kernel(float2 *rope, int32_t max_seq, int32_t d, double theta) {
    const int half = d / 2;
    const int64_t n = (int64_t)max_seq * half;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int pos = (int)(i / half), k = (int)(i % half);
        const double ang = (double)pos * pow(theta, -2.0 * (double)k / (double)d);
        double s, c;
        sincos(ang, &s, &c);
        rope[i] = make_float2((float)c, (float)s);
    }
}

__global__ void greedy_next_kernel(const float *logits, int32_t V, int32_t *tokens, int32_t *positions) {
    const int b = blockIdx.x;
    const float *row = logits + (int64_t)b * V;
    float best = -INFINITY;
    int32_t idx = 0x7FFFFFFF;
    for (int32_t v = threadIdx.x; v < V; v += blockDim.x) {
        const float x = row[v];
        if (x > best) {  // strictly greater: the lowest index wins ties
            best = x;
            idx = v;
        }
    }
    __shared__ float sb[32];
    __shared__ int32_t si[32];
    for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
        if (ob > best || (ob == best && oi < idx)) {
            best = ob;
            idx = oi;
        }
    }
    if ((threadIdx.x & 31) == 0) {
        sb[threadIdx.x >> 5] = best;
        si[threadIdx.x >> 5] = idx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            if (sb[w] > best || (sb[w] == best && si[w] < idx)) {
                best = sb[w];
                idx = si[w];
            }
        tokens[b] = (idx == 0x7FFFFFFF) ? 0 : idx;
        positions[b] += 1;
    }
}

template <int MAXCH>
const void *kernel_ptr() {
    return reinterpret_cast<const void *>(&megakernel<MAXCH>);
}

const void *variant_ptr(int variant) {
    switch (variant) {
        case 2: return kernel_ptr<2>();
        case 4: return kernel_ptr<4>();
        case 8: return kernel_ptr<8>();
        default: return kernel_ptr<16>();
    }
}

}  // namespace

size_t megakernel_smem_bytes(int32_t slot_bytes, int32_t num_slots) {
    return kRingOffset + (size_t)slot_bytes * num_slots;
}

int megakernel_variant(int32_t max_k) {
    const int nch = (max_k / 8 + kComputeThreads - 1) / kComputeThreads;
    if (nch <= 2) return 2;
    if (nch <= 4) return 4;
    if (nch <= 8) return 8;
    return 16;
}

cudaError_t megakernel_set_smem(int variant, size_t smem) {
    return cudaFuncSetAttribute(variant_ptr(variant), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t megakernel_max_active(int variant, size_t smem, int *blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, variant_ptr(variant), kThreads, smem);
}

cudaError_t launch_megakernel(const KParams &p, int variant, int grid, size_t smem, bool cooperative,
                              cudaStream_t stream) {
    void *args[] = {const_cast<KParams *>(&p)};
    if (cooperative)
        return cudaLaunchCooperativeKernel(variant_ptr(variant), dim3(grid), dim3(kThreads), args, smem, stream);
    return cudaLaunchKernel(variant_ptr(variant), dim3(grid), dim3(kThreads), args, smem, stream);
}

cudaError_t launch_rope_table(float2 *rope, int32_t max_seq, int32_t d, float theta, cudaStream_t stream) {
    const int64_t n = (int64_t)max_seq * (d / 2);
    const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    rope_table_kernel<<<grid, 256, 0, stream>>>(rope, max_seq, d, (double)theta);
    return cudaGetLastError();
}

cudaError_t launch_greedy_next(const float *logits, int32_t B, int32_t V, int32_t *tokens, int32_t *positions,
                               cudaStream_t stream) {
    greedy_next_kernel<<<B, 1024, 0, stream>>>(logits, V, tokens, positions);
    return cudaGetLastError();
}

}  // namespace mk
