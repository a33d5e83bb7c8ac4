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

#include <mutex>
#include <type_traits>

#include "mk_kernel.h"
#include "ptx.cuh"

namespace mk {

namespace {

// Attention scratch of one task; the batch-1 matvec reuses the same bytes
// for its per-warp row totals (a CTA runs one task at a time).
struct AttnScratch {
    alignas(16) float q_s[kMaxGroup][kMaxHeadDim];        // RoPE'd, scaled queries (fp32)
    alignas(16) float s_s[kMaxGroup][kAttnStep];          // scores of one step (up to two 64-token blocks)
    alignas(16) uint16_t q_hl[2 * kMaxGroup][kQhlStride];  // queries as bf16 high parts, then low parts
    alignas(16) uint16_t p_hl[2 * kMaxGroup][kPhlStride];  // softmax weights, bf16 high then low parts
};

// Row groups (of at most 8 output values) whose per-warp totals a batch-1
// matvec task keeps in shared memory before one barrier finishes them.
constexpr int kPartGroups = 48;

struct SmemCtl {
    uint64_t full[kMaxSlots];
    uint64_t empty[kMaxSlots];
    uint32_t ready;      // tasks [0, ready) of the queue have their dependencies met
    uint32_t abort;      // local abort flag
    uint32_t last_flag;  // attention: this CTA finished the last split of a head
    uint32_t pad0;
    // dynamic dispatch: the tasks this CTA's scheduler claimed, a ring of
    // task indices (the i-th claimed task in slot i % kJitRing)
    uint32_t jq[kJitRing];
    uint32_t jmma;  // dynamic dispatch: claims the MMA warp has read
    uint32_t jclaimed;   // tasks claimed so far
    uint32_t jdone;      // 1 once every stage is exhausted (jclaimed is final)
    uint32_t jprod;      // claimed tasks the producer has read
    uint32_t jcomp;      // claimed tasks the compute warps have read
    float rms_part[kComputeWarps];
    unsigned long long amax_part[kComputeWarps];  // fused greedy pick: each warp's packed maximum
    float att_m[kMaxGroup], att_l[kMaxGroup], att_alpha[kMaxGroup];
    float att_inv_l[kMaxGroup];
    float merge_w[kMaxSplits][kMaxGroup];  // live split j's weight exp(m_j - max m) in the merge
    float merge_l[kMaxSplits][kMaxGroup];  // live split j's sum of exponentials
    float resid[kMaxResid];                // residual rows of an O / down task, read at task start
    union {
        AttnScratch at;
        alignas(16) float mv_part[kPartGroups][8][kComputeWarps];  // [group][value][warp]
    };
    int32_t mv_grow[kPartGroups];  // first output row of each waiting group
    int32_t mv_gn[kPartGroups];    // rows in it
    float att_pnew[kMaxGroup];                             // weight of the new token
    alignas(16) uint16_t knew[kMaxHeadDim];
    alignas(16) uint16_t vnew[kMaxHeadDim];
    // batched (tensor-core) path
    uint64_t afull[kMaxASlots];   // activation ring
    uint64_t aempty[kMaxASlots];
    uint64_t acc_full[2];         // TMEM accumulator buffers: MMA issuer -> epilogue
    uint64_t acc_empty[2];        // epilogue -> MMA issuer
    uint64_t mma_done;            // drain of the MMA pipe at exit
    uint32_t tmem_base;
    uint32_t ep_last;             // the epilogue finishes this row tile (last contributor)
    float rs[kTcMaxBatch];        // 1/rms of each sequence's projection input
    unsigned long long amax_seq[kTcMaxBatch];  // fused greedy pick: this CTA's packed maximum per sequence
    float ssq_red[4][kTcMaxBatch];  // per-epilogue-warp partial sums of x^2
};

static_assert(sizeof(float) * kPartGroups * 8 * kComputeWarps <= sizeof(AttnScratch),
              "the matvec row totals must fit in the attention scratch they share");

// The rings start at the first 1024-byte boundary after the control block
// (the 128-byte-swizzled TMA tiles of the batched path need that alignment);
// kRingOffset budgets for the worst placement of the dynamic window.
constexpr size_t kRingOffset = (sizeof(SmemCtl) + 1023) / 1024 * 1024 + 1024;
constexpr uint32_t kReadyAbort = 0x7FFFFFFFu;

struct Ctx {
    const KParams *p;
    SmemCtl *sc;
    uint8_t *ring;   // weight / KV ring
    uint8_t *aring;  // activation ring (batched path)
    int cta;
};

// A logit and its row as one 64-bit word whose unsigned order is the pick's:
// the larger logit, then the lower row.  Only finite values and +inf take
// part (as in a strictly-greater scan from -inf, NaN never wins); 0 means
// no candidate.
__device__ __forceinline__ unsigned long long pack_logit(float x, int32_t row) {
    if (!(x > -INFINITY)) return 0ull;
    const uint32_t u = __float_as_uint(x);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)row);
}

__device__ __forceinline__ bool is_proj(int op) { return op == OP_QKV || op == OP_O || op == OP_GU || op == OP_DOWN || op == OP_LM; }

// ------------------------------------------------------ batched-path tiles
// Tensor maps (128 bytes each): per layer wq, wk, wv, wo, w_gate, w_up,
// w_down; then the LM head and the three activation operands.
constexpr int kTmPerLayer = 7;
enum TmIdx : int { TM_WQ = 0, TM_WK, TM_WV, TM_WO, TM_WG, TM_WU, TM_WD };

__device__ __forceinline__ const void *tmap(const KParams &p, int idx) { return p.tmaps + (size_t)idx * 128; }
__device__ __forceinline__ int tm_lm(const KParams &p) { return p.L * kTmPerLayer; }
__device__ __forceinline__ int tm_xa(const KParams &p) { return p.L * kTmPerLayer + 1; }
__device__ __forceinline__ int tm_attn(const KParams &p) { return p.L * kTmPerLayer + 2; }
__device__ __forceinline__ int tm_h(const KParams &p) { return p.L * kTmPerLayer + 3; }

// Activation operand (tensor map) of a projection.
__device__ __forceinline__ int act_map(const KParams &p, int op) {
    return op == OP_O ? tm_attn(p) : (op == OP_DOWN ? tm_h(p) : tm_xa(p));
}

// Weight tensor map and local row tile of row tile `tile` of a projection
// (matrix m = 1 is w_up of gate/up).
__device__ __forceinline__ int weight_map(const KParams &p, int op, int layer, int tile, int m, int *ltile) {
    *ltile = tile;
    switch (op) {
        case OP_QKV: {
            const TcGeom &g = p.tcg[OP_QKV];
            if (tile < g.tiles_q) return layer * kTmPerLayer + TM_WQ;
            if (tile < g.tiles_q + g.tiles_k) {
                *ltile = tile - g.tiles_q;
                return layer * kTmPerLayer + TM_WK;
            }
            *ltile = tile - g.tiles_q - g.tiles_k;
            return layer * kTmPerLayer + TM_WV;
        }
        case OP_O: return layer * kTmPerLayer + TM_WO;
        case OP_GU: return layer * kTmPerLayer + (m ? TM_WU : TM_WG);
        case OP_DOWN: return layer * kTmPerLayer + TM_WD;
        default: return tm_lm(p);
    }
}

// Which range (0 .. n-1) owns unit u when `units` units are cut into n
// balanced contiguous ranges [c*U/n, (c+1)*U/n).
__device__ __forceinline__ int32_t range_of(int64_t u, int64_t units, int64_t n) {
    return (int32_t)(((u + 1) * n - 1) / units);
}
__device__ __forceinline__ int64_t range_start(int64_t c, int64_t units, int64_t n) { return c * units / n; }
// With fewer units than ranges some ranges are empty (and have no task).
__device__ __forceinline__ bool range_nonempty(int64_t c, int64_t units, int64_t n) {
    return range_start(c + 1, units, n) > range_start(c, units, n);
}

// Split-bf16 activation operand [2 * npad][K]: row b holds bf16(v), row
// npad + b holds bf16(v - bf16(v)).  One MMA with N = 2 * npad multiplies
// both halves; their sum keeps about 16 significant bits of v.
__device__ __forceinline__ void store_split(uint16_t *buf, int32_t K, int32_t npad, int32_t b, int64_t col, float v) {
    const uint16_t hi = f32_to_bf16_bits(v);
    const uint16_t lo = f32_to_bf16_bits(v - __uint_as_float((uint32_t)hi << 16));
    buf[(int64_t)b * K + col] = hi;
    buf[(int64_t)(npad + b) * K + col] = lo;
}

// 16 columns of a split accumulator: the high-part columns at `taddr` plus
// the low-part columns npad further on.
__device__ __forceinline__ void tmem_ld_split16(uint32_t taddr, int32_t npad, float (&v)[16]) {
    float lo[16];
    tmem_ld16(taddr, v);
    tmem_ld16(taddr + (uint32_t)npad, lo);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += lo[i];
}

__device__ __forceinline__ bool task_active(const KParams &p, const Task &t) {
    if (p.only_op >= 0) return t.op == p.only_op && t.layer == p.only_layer;
    if (p.skip_lm && t.op == OP_LM) return false;
    return true;
}

__device__ __forceinline__ uint64_t *trace_slot(const KParams &p, int task) {
    return (p.trace && !p.jit) ? p.trace + ((size_t)blockIdx.x * p.trace_stride + task) * 8 : nullptr;
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
// The abort flags and the time budget are checked every kAbortCheckNs only:
// the grid-wide flag is a global-memory load whose latency would otherwise
// sit between a phase completing and the waiter noticing it.
constexpr uint64_t kAbortCheckNs = 20000;

__device__ bool wait_mbar(const Ctx &c, uint64_t *bar, uint32_t parity, int32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint64_t next = t0 + kAbortCheckNs;
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
        const uint64_t now = globaltimer_ns();
        if (now >= next) {
            if (local_abort(c) || global_abort(*c.p)) {
                set_local_abort(c);
                return false;
            }
            if (now - t0 > c.p->timeout_ns) {
                record_error(c, 4 /*MK_ERR_TIMEOUT*/, site, (int32_t)parity);
                return false;
            }
            next = now + kAbortCheckNs;
        }
    }
}

// Dynamic dispatch: the i-th task this CTA's scheduler claimed.  Waits
// (bounded) until it is claimed; false once every stage is exhausted and i
// is past the last claim, or on abort or timeout (the CTA is then aborted).
// The reader publishes i + 1 in *seen once it holds the task, so the
// scheduler may reuse the ring slot.
__device__ __noinline__ bool jit_task(const Ctx &c, int i, Task *t, uint32_t *seen) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if ((uint32_t)i < ld_acquire_cta(&c.sc->jclaimed)) break;
        if (ld_acquire_cta(&c.sc->jdone) && (uint32_t)i >= ld_acquire_cta(&c.sc->jclaimed)) return false;
        if ((it & 63u) == 0) {
            if (local_abort(c)) return false;
            if (globaltimer_ns() - t0 > 4 * c.p->timeout_ns) {
                record_error(c, 4 /*MK_ERR_TIMEOUT*/, SITE_READY_WAIT, i);
                return false;
            }
        }
    }
    *t = c.p->tasks[c.sc->jq[i % kJitRing]];
    if (seen) st_release_cta(seen, (uint32_t)(i + 1));
    return true;
}

// ----------------------------------------------------------------- pages
// A task's immutable operands are cut into ring-slot "pages"; producer and
// consumers enumerate them with the same loops.

// matrix and local row of operator row `row` (w: the layer's pointers, held
// in registers by the caller)
__device__ __forceinline__ const uint16_t *mv_matrix(const KParams &p, int op, const LayerW &w, int32_t row,
                                                     int32_t *local) {
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
    int32_t pos;       // position of the new token
    int32_t ctx;       // positions read from the cache: [0, ctx)
    int32_t blo, bhi;  // 64-token blocks [blo, bhi) of [0, ctx)
    bool has_new;      // this split also attends to the new token, from registers
    int32_t n_live;    // splits of this (sequence, kv head) with any work
};

// The cached context [0, ctx) is cut into aligned 64-token blocks, and split
// s of S takes blocks [s*nb/S, (s+1)*nb/S).  ctx = pos when the last split
// handles the new token at pos itself (not read from the cache); ctx =
// pos + 1 in kv-append graphs, where OP_KVA put it in the cache first.
__device__ __forceinline__ AttnRange attn_range(const KParams &p, const Task &t) {
    AttnRange r;
    r.pos = p.positions[(int64_t)t.a0 * p.pos_stride];
    r.ctx = p.kv_appended ? r.pos + 1 : r.pos;
    const int64_t nb = (r.ctx + kAttnBlock - 1) / kAttnBlock;
    r.blo = (int32_t)((int64_t)t.a2 * nb / t.a3);
    r.bhi = (int32_t)((int64_t)(t.a2 + 1) * nb / t.a3);
    r.has_new = !p.kv_appended && (t.a2 == t.a3 - 1);
    // nb <= S blocks land on nb distinct splits (the last one among them);
    // with no cached block only the new token's split works
    r.n_live = nb < 1 ? 1 : (nb < t.a3 ? (int32_t)nb : t.a3);
    return r;
}

// The j-th of the n_live splits with work over a cached context of ctx
// positions (cached blocks, or the new token: the last split).  With nb <= S
// blocks, block j is the only block of split ((j + 1) S - 1) / nb; with more
// blocks every split has some.
__device__ __forceinline__ int32_t live_split(int32_t ctx, int32_t j, int32_t S) {
    const int64_t nb = (ctx + kAttnBlock - 1) / kAttnBlock;
    if (nb == 0) return S - 1;
    if (nb > S) return j;
    return (int32_t)(((int64_t)(j + 1) * S - 1) / nb);
}

__device__ __forceinline__ int64_t kv_offset(const KParams &p, int layer, int32_t page, int32_t kvh, int32_t slot) {
    return (((int64_t)layer * p.num_pages + page) * p.nkv + kvh) * (int64_t)p.page_size * p.d + (int64_t)slot * p.d;
}

// ------------------------------------------------------------- producer

struct Producer {
    uint32_t issued = 0;
    // slot index and phase bit of ring slot number `issued`, advanced with it
    // (one single-thread loop: no division per slot)
    uint32_t si = 0, sph = 0;
    uint64_t pol;
    uint64_t *tr = nullptr;  // trace entry of the current task
    uint32_t ns = 0;         // ring slots (kept in a register)
    uint32_t slot_bytes = 0;
    uint32_t fmax = 0;       // copies in flight at most (0: every free slot)

    // Every call is followed by exactly one ++issued once the slot's copies
    // are issued; si and sph move on here.
    __device__ bool acquire_slot(const Ctx &c, uint32_t *slot) {
        const uint32_t s = si;
        const uint64_t t0 = tr ? globaltimer_ns() : 0;
        if (!wait_mbar(c, &c.sc->empty[s], sph ^ 1u, SITE_EMPTY_WAIT)) return false;
        if (fmax != 0 && issued >= fmax) {
            // copy number issued - fmax must have landed: fewer bytes queued
            // in the memory system ahead of this SM's other requests, and a
            // gpu-scope fence (which waits for this SM's copies in flight)
            // stays short.  fmax < ns: that copy is in this round or the last.
            const uint32_t ks = (s >= fmax) ? s - fmax : s + ns - fmax;
            const uint32_t kph = (s >= fmax) ? sph : (sph ^ 1u);
            if (!wait_mbar(c, &c.sc->full[ks], kph, SITE_EMPTY_WAIT)) return false;
        }
        if (++si == ns) {
            si = 0;
            sph ^= 1u;
        }
        if (tr) {
            const uint64_t t1 = globaltimer_ns();
            if (tr[4] == 0) tr[4] = t1;
            tr[5] += t1 - t0;
        }
        *slot = s;
        return true;
    }

    // Starts ring slot number `issued`, which will receive `bytes` bytes:
    // waits for a free slot (and the in-flight cap) and arms its full
    // barrier.  False on abort or timeout.
    __device__ __forceinline__ bool begin_slot(const Ctx &c, uint32_t *slot, uint32_t bytes) {
        if (!acquire_slot(c, slot)) return false;
        mbar_arrive_expect_tx(&c.sc->full[*slot], bytes);
        return true;
    }
    // One contiguous piece of a slot.
    __device__ __forceinline__ void copy(const Ctx &c, uint32_t s, uint8_t *dst, const void *src, uint32_t bytes) {
        bulk_g2s(dst, src, bytes, &c.sc->full[s], pol);
    }

    __device__ bool run_matvec(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const int op = t.op;
        const MvGeom g = p.mv[op];              // register copies: the copy loop's
        const LayerW lw = p.layers[t.layer];    // inline asm must not force reloads
        const int32_t qb1 = p.nq * p.d, qb2 = qb1 + p.nkv * p.d, qb3 = p.qkv_rows;
        for (int32_t row = t.a0; row < t.a1;) {
            int32_t n = min(g.rpp, t.a1 - row);
            if (op == OP_QKV) n = min(n, (row < qb1 ? qb1 : (row < qb2 ? qb2 : qb3)) - row);
            int32_t lr;
            const uint16_t *W = mv_matrix(p, op, lw, row, &lr);
            if (g.rps == 8 && g.row_mult == 2) {
                // gate rows and up rows of the group in one slot: two contiguous copies
                uint32_t s;
                const uint32_t bytes = (uint32_t)(n * g.K * 2);
                if (!begin_slot(c, &s, 2 * bytes)) return false;
                uint8_t *dst = c.ring + (size_t)s * slot_bytes;
                copy(c, s, dst, W + (int64_t)lr * g.K, bytes);
                copy(c, s, dst + (size_t)4 * g.K * 2, lw.w_up + (int64_t)lr * g.K, bytes);
                ++issued;
                row += n;
                continue;
            }
            if (g.rps > 0) {
                // whole-row slots: rps rows of one matrix, one contiguous copy each
                for (int m = 0; m < g.row_mult; ++m) {
                    const uint16_t *Wm = (m == 0) ? W : lw.w_up;
                    for (int32_t j0 = 0; j0 < n; j0 += g.rps) {
                        const int32_t cnt = min(g.rps, n - j0);
                        uint32_t s;
                        const uint32_t bytes = (uint32_t)(cnt * g.K * 2);
                        if (!begin_slot(c, &s, bytes)) return false;
                        copy(c, s, c.ring + (size_t)s * slot_bytes, Wm + (int64_t)(lr + j0) * g.K, bytes);
                        ++issued;
                    }
                }
                row += n;
                continue;
            }
            if (g.ksplit > kMvResident) return run_matvec_long(c, t, g, lw, row);
            for (int32_t ks = 0; ks < g.ksplit; ++ks) {
                const int32_t k0 = ks * g.kc;
                const int32_t pw = min(g.kc, g.K - k0);
                const uint32_t bytes = (uint32_t)(g.row_mult * n * pw * 2);
                uint32_t s;
                if (!begin_slot(c, &s, bytes)) return false;
                uint8_t *dst = c.ring + (size_t)s * slot_bytes;
                for (int m = 0; m < g.row_mult; ++m) {
                    const uint16_t *Wm = (m == 0) ? W : lw.w_up;
                    if (g.ksplit == 1) {
                        copy(c, s, dst + (size_t)m * n * pw * 2, Wm + (int64_t)lr * g.K, (uint32_t)(n * pw * 2));
                    } else {
                        for (int32_t r = 0; r < n; ++r)
                            copy(c, s, dst + (size_t)(m * n + r) * pw * 2, Wm + (int64_t)(lr + r) * g.K + k0,
                                 (uint32_t)(pw * 2));
                    }
                }
                ++issued;
            }
            row += n;
        }
        return true;
    }

    // Rows of inputs longer than kMvResident pieces, from `row` on: up to
    // kMvSuper row groups at a time, piece by piece (piece ks of every group
    // of the super-group, then piece ks + 1), the order in which the compute
    // warps consume them, so that each input piece they load from L2 serves
    // every group of the super-group.  A slot holds piece ks of one group's
    // rows (gate rows, then up rows), one bulk copy per row.
    __device__ bool run_matvec_long(const Ctx &c, const Task &t, const MvGeom &g, const LayerW &lw, int32_t row) {
        const KParams &p = *c.p;
        const int op = t.op;
        const int32_t qb1 = p.nq * p.d, qb2 = qb1 + p.nkv * p.d, qb3 = p.qkv_rows;
        while (row < t.a1) {
            int32_t gr[kMvSuper], gn[kMvSuper];
            int ng = 0;
            for (int32_t r = row; ng < kMvSuper && r < t.a1; ++ng) {
                int32_t n = min(g.rpp, t.a1 - r);
                if (op == OP_QKV) n = min(n, (r < qb1 ? qb1 : (r < qb2 ? qb2 : qb3)) - r);
                gr[ng] = r;
                gn[ng] = n;
                r += n;
            }
            for (int32_t ks = 0; ks < g.ksplit; ++ks) {
                const int32_t k0 = ks * g.kc;
                const int32_t pw = min(g.kc, g.K - k0);
                if (op == OP_DOWN && p.down_maps != nullptr) {
                    // one 3-D TMA copy per slot: piece ks of rpp rows (rows
                    // past the group's own belong to the next group or read as 0)
                    const void *map = p.down_maps + (size_t)t.layer * 128;
                    for (int gi = 0; gi < ng; ++gi) {
                        uint32_t s;
                        if (!begin_slot(c, &s, (uint32_t)(g.rpp * g.kc * 2))) return false;
                        tma_load_3d(c.ring + (size_t)s * slot_bytes, map, 0, k0 / 256, gr[gi], &c.sc->full[s], pol);
                        ++issued;
                    }
                    continue;
                }
                for (int gi = 0; gi < ng; ++gi) {
                    const int32_t n = gn[gi];
                    uint32_t s;
                    if (!begin_slot(c, &s, (uint32_t)(g.row_mult * n * pw * 2))) return false;
                    int32_t lr;
                    const uint16_t *W = mv_matrix(p, op, lw, gr[gi], &lr);
                    uint8_t *dst = c.ring + (size_t)s * slot_bytes;
                    for (int m = 0; m < g.row_mult; ++m) {
                        const uint16_t *Wm = (m == 0) ? W : lw.w_up;
                        for (int32_t r = 0; r < n; ++r)
                            copy(c, s, dst + (size_t)(m * n + r) * pw * 2, Wm + (int64_t)(lr + r) * g.K + k0,
                                 (uint32_t)(pw * 2));
                    }
                    ++issued;
                }
            }
            row = gr[ng - 1] + gn[ng - 1];
        }
        return true;
    }

    // Batch 1, on reaching an O projection task: while the attention phase
    // holds the compute warps, the ring fills with O rows and the weight
    // stream would stop.  Prefetch into L2 (up to l2_prefetch_bytes) the O
    // rows the ring cannot hold, then the first gate/up rows of the next
    // task, so that HBM keeps working and those copies later hit L2.
    __device__ void prefetch_past_attention(const Ctx &c, const Task &t, const Task *next) {
        const KParams &p = *c.p;
        int64_t budget = p.l2_prefetch_bytes;
        const int64_t ring = (int64_t)ns * slot_bytes;
        const int64_t rowb_o = (int64_t)p.mv[OP_O].K * 2;
        const char *ob = reinterpret_cast<const char *>(p.layers[t.layer].wo) + (int64_t)t.a0 * rowb_o;
        const int64_t obytes = (int64_t)(t.a1 - t.a0) * rowb_o;
        for (int64_t off = ring; off < obytes && budget > 0; off += 32768) {
            const int64_t n = min(min((int64_t)32768, obytes - off), budget);
            prefetch_l2(ob + off, (uint32_t)n);
            budget -= n;
        }
        if (next == nullptr || next->op != OP_GU || !task_active(p, *next) || budget <= 0) return;
        const int64_t rowb = (int64_t)p.mv[OP_GU].K * 2;
        const int64_t rows = min((int64_t)(next->a1 - next->a0), budget / (2 * rowb));
        const LayerW &lw = p.layers[next->layer];
        const char *gb = reinterpret_cast<const char *>(lw.w_gate) + (int64_t)next->a0 * rowb;
        const char *ub = reinterpret_cast<const char *>(lw.w_up) + (int64_t)next->a0 * rowb;
        for (int64_t off = 0; off < rows * rowb; off += 32768) {
            const uint32_t n = (uint32_t)min((int64_t)32768, rows * rowb - off);
            prefetch_l2(gb + off, n);
            prefetch_l2(ub + off, n);
        }
    }

    // KV of one 64-token block: TMA tiles of ts tokens x 64 columns (128-byte
    // swizzle) from the paged pools, K halves then V halves, in 64/ts slots.
    __device__ bool run_attn(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const AttnRange r = attn_range(p, t);
        const int ts = p.attn_ts, halves = p.d / 64;
        const int32_t *pt = p.page_table + (int64_t)t.a0 * p.pt_stride;
        for (int32_t blk = r.blo; blk < r.bhi; ++blk) {
            const int32_t tok0 = blk * kAttnBlock;
            const int32_t pg = pt[tok0 / p.page_size];
            const int32_t row0 =
                (int32_t)((((int64_t)t.layer * p.num_pages + pg) * p.nkv + t.a1) * p.page_size + tok0 % p.page_size);
            for (int j = 0; j < kAttnBlock / ts; ++j) {
                uint32_t s;
                if (!begin_slot(c, &s, (uint32_t)(2 * halves * ts * 128))) return false;
                uint8_t *dst = c.ring + (size_t)s * slot_bytes;
                if (p.kv_halves_3d) {
                    tma_load_3d(dst, p.kv_maps[0], 0, row0 + j * ts, 0, &c.sc->full[s], pol);
                    tma_load_3d(dst + (size_t)halves * ts * 128, p.kv_maps[1], 0, row0 + j * ts, 0, &c.sc->full[s],
                                pol);
                    ++issued;
                    continue;
                }
                for (int h = 0; h < halves; ++h) {
                    tma_load_2d(dst + (size_t)h * ts * 128, p.kv_maps[0], h * 64, row0 + j * ts, &c.sc->full[s], pol);
                    tma_load_2d(dst + (size_t)(halves + h) * ts * 128, p.kv_maps[1], h * 64, row0 + j * ts,
                                &c.sc->full[s], pol);
                }
                ++issued;
            }
        }
        return true;
    }

    // Batched path: one unit of 128 rows x tc_sub 64-column sub-tiles per
    // slot by TMA, one copy per sub-tile (two units for gate/up: the gate
    // tile, then the matching up tile).
    __device__ bool run_gemm(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const TcGeom &g = p.tcg[t.op];
        const int mats = (t.op == OP_GU) ? 2 : 1;
        const int sub = p.tc_sub;
        for (int32_t u = t.a0; u < t.a1; ++u) {
            const int32_t tile = u / g.kchunks, kc = u % g.kchunks;
            for (int m = 0; m < mats; ++m) {
                uint32_t s;
                if (!acquire_slot(c, &s)) return false;
                int lt;
                const int map = weight_map(p, t.op, t.layer, tile, m, &lt);
                mbar_arrive_expect_tx(&c.sc->full[s], slot_bytes);
                for (int j = 0; j < sub; ++j)
                    tma_load_2d(c.ring + (size_t)s * slot_bytes + (size_t)j * kTcTileM * kTcTileK * 2, tmap(p, map),
                                (kc * sub + j) * kTcTileK, lt * kTcTileM, &c.sc->full[s], pol);
                ++issued;
            }
        }
        return true;
    }

    // Kv-append graphs: the cache blocks an attention task reads include
    // positions that OP_KVA tasks write in this launch, so their copies wait
    // until the scheduler has seen the task's event (queue position i
    // released), then order those generic-proxy writes before the TMA reads.
    __device__ bool wait_released(const Ctx &c, int i) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            const uint32_t r = ld_acquire_cta(&c.sc->ready);
            if (r == kReadyAbort) return false;
            if (r >= (uint32_t)(i + 1)) break;
            if ((it & 63u) == 0) {
                if (local_abort(c)) return false;
                if (globaltimer_ns() - t0 > 4 * c.p->timeout_ns) {
                    record_error(c, 4 /*MK_ERR_TIMEOUT*/, SITE_READY_WAIT, i);
                    return false;
                }
            }
        }
        fence_proxy_async_global();
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

template <bool JIT>
__device__ void producer_role(const Ctx &c, const Task *q, int nt) {
    if ((threadIdx.x & 31) != 0) return;
    Producer pr;
    pr.pol = policy_evict_first();
    pr.ns = (uint32_t)c.p->num_slots;
    pr.slot_bytes = (uint32_t)c.p->slot_bytes;
    pr.fmax = (c.p->max_inflight > 0 && (uint32_t)c.p->max_inflight < pr.ns) ? (uint32_t)c.p->max_inflight : 0u;
    for (int i = 0;; ++i) {
        Task t;
        if (JIT) {
            if (!jit_task(c, i, &t, &c.sc->jprod)) break;
        } else {
            if (i >= nt) break;
            t = q[i];
        }
        if (!task_active(*c.p, t)) continue;
        pr.tr = trace_slot(*c.p, i);
        bool ok = true;
        if (t.op == OP_O && !c.p->tc && c.p->l2_prefetch_bytes > 0 && !JIT)
            pr.prefetch_past_attention(c, t, i + 1 < nt ? &q[i + 1] : nullptr);
        if (t.op == OP_ATTN) ok = (!c.p->kv_appended || pr.wait_released(c, i)) && pr.run_attn(c, t);
        else if (t.op == OP_EMBED || t.op == OP_KVA) ok = true;
        else ok = c.p->tc ? pr.run_gemm(c, t) : pr.run_matvec(c, t);
        if (!ok) break;
    }
    pr.drain(c);
}

// ------------------------------------------------------------ scheduler

// Batched path: after a projection task's event fires, the scheduler streams
// its activation operand (npad rows x 64 columns per unit, bf16, written
// earlier in this launch by other CTAs) into the activation ring.
struct ActProducer {
    uint32_t issued = 0;
    uint32_t si = 0, sph = 0;  // slot index and phase bit of activation slot number `issued`
    uint64_t pol;

    __device__ bool run(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const TcGeom &g = p.tcg[t.op];
        const void *map = tmap(p, act_map(p, t.op));
        const uint32_t ns = (uint32_t)p.num_aslots;
        fence_proxy_async_global();  // generic-proxy writes (ordered by the acquire) -> TMA reads
        int32_t kc = t.a0 % g.kchunks;
        for (int32_t u = t.a0; u < t.a1; ++u) {
            const uint32_t s = si;
            if (!wait_mbar(c, &c.sc->aempty[s], sph ^ 1u, SITE_EMPTY_WAIT)) return false;
            mbar_arrive_expect_tx(&c.sc->afull[s], (uint32_t)p.aslot_bytes);
            for (int j = 0; j < p.tc_sub; ++j)
                tma_load_2d(c.aring + (size_t)s * p.aslot_bytes + (size_t)j * (p.aslot_bytes / p.tc_sub), map,
                            (kc * p.tc_sub + j) * kTcTileK, 0, &c.sc->afull[s], pol);
            ++issued;
            if (++si == ns) {
                si = 0;
                sph ^= 1u;
            }
            if (++kc == g.kchunks) kc = 0;
        }
        return true;
    }

    __device__ void drain(const Ctx &c) {
        const uint32_t ns = (uint32_t)c.p->num_aslots;
        const uint32_t lim = issued < ns ? issued : ns;
        for (uint32_t s = 0; s < lim; ++s) {
            const uint32_t k = issued - 1 - ((issued - 1 - s) % ns);
            const uint32_t par = (k / ns) & 1u;
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&c.sc->afull[s], par)) {
                if (globaltimer_ns() - t0 > c.p->timeout_ns) {
                    record_error(c, 4, SITE_DRAIN_WAIT, (int32_t)s);
                    break;
                }
            }
        }
    }
};

__device__ void scheduler_loop(const Ctx &c, const Task *q, int nt, ActProducer &ap) {
    const KParams &p = *c.p;
    const bool use_events = p.only_op < 0;
    for (int i = 0; i < nt; ++i) {
        const Task t = q[i];
        if (use_events && task_active(p, t) && t.wait_ev != kNoEvent) {
            const uint32_t *ctr = p.ctl + t.wait_ev;
            if (ld_acquire_gpu(ctr) < t.wait_count) {
                const uint64_t t0 = globaltimer_ns();
                uint64_t next = t0 + kAbortCheckNs;
                for (;;) {
                    // relaxed polls; one acquire once the count is seen
                    if (ld_relaxed_gpu(ctr) >= t.wait_count && ld_acquire_gpu(ctr) >= t.wait_count) break;
                    const uint64_t now = globaltimer_ns();
                    if (now >= next) {
                        if (local_abort(c) || global_abort(p)) {
                            set_local_abort(c);
                            st_release_cta(&c.sc->ready, kReadyAbort);
                            return;
                        }
                        if (now - t0 > p.timeout_ns) {
                            record_error(c, 4, SITE_EVENT_WAIT, t.wait_ev);
                            st_release_cta(&c.sc->ready, kReadyAbort);
                            return;
                        }
                        next = now + kAbortCheckNs;
                    }
                }
            }
        }
        if (uint64_t *tr = trace_slot(p, i)) tr[0] = globaltimer_ns();
        st_release_cta(&c.sc->ready, (uint32_t)(i + 1));
        if (p.tc && is_proj(t.op) && task_active(p, t) && !ap.run(c, t)) {
            st_release_cta(&c.sc->ready, kReadyAbort);
            return;
        }
    }
}

// Dynamic dispatch.  The scheduler claims tasks for its CTA at run time:
// the next unclaimed task of the earliest stage with any left (one relaxed
// atomicAdd on the stage's claim counter), as long as fewer than kJitRing
// claimed tasks are ahead of the producer and the compute warps; then it
// releases them in claim order once their events reach their thresholds,
// claiming more while it waits (a ring slot is reused only once the
// producer and the compute warps have read its task and the scheduler has
// released it).  Every task of a stage is claimed before any
// task of the next, and each CTA runs its claims in order, so a stage's
// tasks never wait on a later stage's: the run cannot deadlock.
__device__ __noinline__ void scheduler_loop_jit(const Ctx &c, ActProducer &ap) {
    const KParams &p = *c.p;
    SmemCtl *sc = c.sc;
    uint32_t claimed = 0, released = 0;
    int32_t stage = 0;
    bool done = false;
    auto try_claim = [&]() -> bool {
        while (stage < p.n_stages) {
            // a slot is free once the producer and the compute warps have
            // read its task and this scheduler has released it
            const uint32_t jcomp = ld_acquire_cta(&sc->jcomp);
            uint32_t behind = min(min(ld_acquire_cta(&sc->jprod), jcomp), released);
            if (p.tc) behind = min(behind, ld_acquire_cta(&sc->jmma));
            if (claimed - behind >= (uint32_t)kJitRing) return false;
            // claim only kJitAhead tasks beyond the one the compute warps hold:
            // a CTA that claimed far ahead would keep later stages' tasks from
            // the idle CTAs, and one claim ahead lets the producer stream the
            // next task's weights
            if (claimed >= jcomp + (uint32_t)kJitAhead) return false;
            const int32_t s0 = p.stage_off[stage], n = p.stage_off[stage + 1] - s0;
            const uint32_t idx = atomicAdd(p.ctl + p.cl.claim_idx + stage, 1u);
            if (idx < (uint32_t)n) {
                sc->jq[claimed % kJitRing] = (uint32_t)(s0 + (int32_t)idx);
                st_release_cta(&sc->jclaimed, ++claimed);
                return true;
            }
            ++stage;
        }
        if (!done) {
            st_release_cta(&sc->jdone, 1u);
            done = true;
        }
        return false;
    };
    const uint64_t t_start = globaltimer_ns();
    uint64_t next = t_start + kAbortCheckNs;
    for (;;) {
        while (try_claim()) {
        }
        if (released < claimed) {
            const Task t = p.tasks[sc->jq[released % kJitRing]];
            if (t.wait_ev != kNoEvent) {
                const uint32_t *ctr = p.ctl + t.wait_ev;
                const uint64_t t0 = globaltimer_ns();
                uint64_t nx = t0 + kAbortCheckNs;
                while (!(ld_relaxed_gpu(ctr) >= t.wait_count && ld_acquire_gpu(ctr) >= t.wait_count)) {
                    try_claim();
                    const uint64_t now = globaltimer_ns();
                    if (now >= nx) {
                        if (local_abort(c) || global_abort(p)) {
                            set_local_abort(c);
                            st_release_cta(&sc->ready, kReadyAbort);
                            return;
                        }
                        if (now - t0 > p.timeout_ns) {
                            record_error(c, 4, SITE_EVENT_WAIT, t.wait_ev);
                            st_release_cta(&sc->ready, kReadyAbort);
                            return;
                        }
                        nx = now + kAbortCheckNs;
                    }
                }
            }
            st_release_cta(&sc->ready, ++released);
            if (p.tc && is_proj(t.op) && !ap.run(c, t)) {
                st_release_cta(&sc->ready, kReadyAbort);
                return;
            }
            next = globaltimer_ns() + kAbortCheckNs;
        } else if (done) {
            return;
        } else {
            // the ring is full of released tasks the compute warps have not taken yet
            const uint64_t now = globaltimer_ns();
            if (now >= next) {
                if (local_abort(c) || global_abort(p)) {
                    set_local_abort(c);
                    st_release_cta(&sc->ready, kReadyAbort);
                    return;
                }
                if (now - t_start > 4 * p.timeout_ns) {
                    record_error(c, 4, SITE_EVENT_WAIT, -1);
                    st_release_cta(&sc->ready, kReadyAbort);
                    return;
                }
                next = now + kAbortCheckNs;
            }
        }
    }
}

template <bool JIT>
__device__ void scheduler_role(const Ctx &c, const Task *q, int nt) {
    if ((threadIdx.x & 31) != 0) return;
    ActProducer ap;
    ap.pol = policy_evict_last();
    if (JIT) scheduler_loop_jit(c, ap);
    else scheduler_loop(c, q, nt, ap);
    if (c.p->tc) ap.drain(c);
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
// Barrier of the compute warps that also ORs a flag over them, so that every
// warp takes the same branch on it.
__device__ __forceinline__ bool compute_bar_or(bool v) { return named_bar_or(1, kComputeThreads, v); }
// Barrier of the four epilogue warps of the batched path.
constexpr int kEpiThreads = kComputeThreads;  // the batched epilogue runs on every compute warp
__device__ __forceinline__ void epi_bar() { named_bar_sync(2, kEpiThreads); }

// Sums 8 per-lane values over the warp and scatters the result: lane l
// returns the warp total of value l/4 (each total lands on 4 lanes).  Halving
// exchanges (16, 8, 4) then two full butterflies: 9 shuffles instead of 40.
__device__ __forceinline__ float warp_reduce8(const float (&a)[8], int lane) {
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
    float b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = h16 ? a[i] : a[i + 4];
        b[i] = (h16 ? a[i + 4] : a[i]) + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
    float c2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = h8 ? b[i] : b[i + 2];
        c2[i] = (h8 ? b[i + 2] : b[i]) + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
    float d = (h4 ? c2[1] : c2[0]) + __shfl_xor_sync(0xFFFFFFFFu, h4 ? c2[0] : c2[1], 4);
    d += __shfl_xor_sync(0xFFFFFFFFu, d, 2);
    d += __shfl_xor_sync(0xFFFFFFFFu, d, 1);
    return d;
}


// Sums 16 per-lane values over the warp and scatters the result: lane l
// returns the warp total of value (l / 2) % 16 (each total lands on 2 lanes).
__device__ __forceinline__ float warp_reduce16(const float (&a)[16], int lane) {
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
    float b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = (h16 ? a[i + 8] : a[i]) + __shfl_xor_sync(0xFFFFFFFFu, h16 ? a[i] : a[i + 8], 16);
    float c4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c4[i] = (h8 ? b[i + 4] : b[i]) + __shfl_xor_sync(0xFFFFFFFFu, h8 ? b[i] : b[i + 4], 8);
    float d2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) d2[i] = (h4 ? c4[i + 2] : c4[i]) + __shfl_xor_sync(0xFFFFFFFFu, h4 ? c4[i] : c4[i + 2], 4);
    float e = (h2 ? d2[1] : d2[0]) + __shfl_xor_sync(0xFFFFFFFFu, h2 ? d2[0] : d2[1], 2);
    e += __shfl_xor_sync(0xFFFFFFFFu, e, 1);
    return e;
}

// Maximum of 16 per-lane 64-bit keys over the warp, scattered: lane l
// returns the warp maximum of key (l / 2) % 16 (the pattern of warp_reduce16).
__device__ __forceinline__ unsigned long long warp_max16_u64(const unsigned long long (&a)[16], int lane) {
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
    auto mx = [](unsigned long long x, unsigned long long y) { return x > y ? x : y; };
    unsigned long long b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = mx(h16 ? a[i + 8] : a[i], __shfl_xor_sync(0xFFFFFFFFu, h16 ? a[i] : a[i + 8], 16));
    unsigned long long c4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c4[i] = mx(h8 ? b[i + 4] : b[i], __shfl_xor_sync(0xFFFFFFFFu, h8 ? b[i] : b[i + 4], 8));
    unsigned long long d2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) d2[i] = mx(h4 ? c4[i + 2] : c4[i], __shfl_xor_sync(0xFFFFFFFFu, h4 ? c4[i] : c4[i + 2], 4));
    unsigned long long e = mx(h2 ? d2[1] : d2[0], __shfl_xor_sync(0xFFFFFFFFu, h2 ? d2[0] : d2[1], 2));
    return mx(e, __shfl_xor_sync(0xFFFFFFFFu, e, 1));
}

// acc (two fp32 lanes, even and odd columns) += the 8 bf16 weights of w
// times x: paired fp32 FMAs (fma.rn.f32x2), one per two weights.  The bf16
// halves of each 32-bit word are widened exactly (shift, mask).
__device__ __forceinline__ void dot8x2(uint64_t &acc, const uint4 w, const float *x) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        asm("{\n\t.reg .b64 wp, xp;\n\t"
            "mov.b64 wp, {%1, %2};\n\t"
            "mov.b64 xp, {%3, %4};\n\t"
            "fma.rn.f32x2 %0, wp, xp, %0;\n\t}"
            : "+l"(acc)
            : "r"(ws[i] << 16), "r"(ws[i] & 0xFFFF0000u), "f"(x[2 * i]), "f"(x[2 * i + 1]));
    }
}

__device__ __forceinline__ float sum_x2(uint64_t acc) {
    return __uint_as_float((uint32_t)acc) + __uint_as_float((uint32_t)(acc >> 32));
}

struct Consumer {
    uint32_t ns = 0;         // ring slots and slot size (kept in registers)
    uint32_t slot_bytes = 0;
    bool tcm = false;        // batched (tensor-core) plan
    uint32_t consumed = 0;   // weight / KV ring slots
    uint32_t aconsumed = 0;  // activation ring slots (batched path)
    uint32_t seg = 0;        // accumulator segments (batched path)
    int ct, wc, lane;  // compute-thread index, compute-warp index, lane
    bool tracing = false;
    uint64_t full_wait_ns = 0;  // traced: waits for filled weight / KV slots
    uint64_t act_wait_ns = 0;   // traced (batched): waits for activation tiles
    uint64_t acc_wait_ns = 0;   // traced (batched): waits for a free TMEM accumulator

    // A failed wait (abort or timeout) marks the CTA aborted but keeps the
    // control flow: all compute warps must reach the same named barriers, so
    // they leave only together, at a task boundary.
    // Wait for ring slot number k (k = consumed + j for lookahead).
    __device__ uint32_t wait_slot_at(const Ctx &c, uint32_t k) {
        const uint32_t s = k % ns;
        const uint64_t t0 = tracing ? globaltimer_ns() : 0;
        wait_mbar(c, &c.sc->full[s], (k / ns) & 1u, SITE_FULL_WAIT);
        if (tracing) full_wait_ns += globaltimer_ns() - t0;
        return s;
    }

    __device__ uint32_t wait_slot(const Ctx &c) { return wait_slot_at(c, consumed); }

    // Batch 1: one arrival per compute warp.  Batched path: the slot's empty
    // barrier also takes MMA commits, so it counts one arrival, made after
    // every compute warp is done with the slot.
    __device__ void release_slot(const Ctx &c, uint32_t s) {
        if (tcm) {
            compute_bar();
            if (ct == 0) mbar_arrive(&c.sc->empty[s]);
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.sc->empty[s]);
        }
        ++consumed;
    }

    // ------------------------------------------------------- matvec task
    // Thread ct owns input chunks ct + 256 j (8 columns each), which are
    // exactly its chunk of row piece j; so every slot costs each thread one
    // 128-bit shared load and 4 paired FMAs per row.  Row sums are kept per
    // thread across the pieces of a row group and reduced once per group.
    // Inputs of at most two pieces (4096 columns) stay normalised in
    // registers for the whole task; longer inputs are re-read per piece from
    // L2 (one piece ahead) and normalised on the fly.
    __device__ void load_piece(const KParams &p, const float *xin, const uint16_t *emb_row, const uint16_t *gain,
                               float r, int32_t nchunk, int ks, float (&v)[8]) const {
        const int32_t ch = ct + kComputeThreads * ks;
        if (ch >= nchunk) {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
            return;
        }
        if (emb_row) {
            const uint4 e = __ldg(reinterpret_cast<const uint4 *>(emb_row) + ch);
            v[0] = bf16_lo(e.x); v[1] = bf16_hi(e.x); v[2] = bf16_lo(e.y); v[3] = bf16_hi(e.y);
            v[4] = bf16_lo(e.z); v[5] = bf16_hi(e.z); v[6] = bf16_lo(e.w); v[7] = bf16_hi(e.w);
        } else {
            const float4 a = ld_cg_f4(xin + ch * 8), b = ld_cg_f4(xin + ch * 8 + 4);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
        if (gain) {
            const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(gain) + ch);
            v[0] *= r * bf16_lo(gv.x); v[1] *= r * bf16_hi(gv.x); v[2] *= r * bf16_lo(gv.y); v[3] *= r * bf16_hi(gv.y);
            v[4] *= r * bf16_lo(gv.z); v[5] *= r * bf16_hi(gv.z); v[6] *= r * bf16_lo(gv.w); v[7] *= r * bf16_hi(gv.w);
        }
    }

    // One ring slot: 8 rows (of which R are live) of the piece held in slot s.
    __device__ __forceinline__ void mv_slot(const Ctx &c, int32_t pw8, int32_t R, const float (&xv)[8],
                                            uint64_t (&acc2)[8]) {
        const uint32_t s = wait_slot(c);
        const uint4 *base = reinterpret_cast<const uint4 *>(c.ring + (size_t)s * slot_bytes) + ct;
        // the slot goes back to the producer as soon as its data is in registers
        uint4 w[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) w[r] = (ct < pw8 && r < R) ? base[r * pw8] : make_uint4(0u, 0u, 0u, 0u);
        release_slot(c, s);
#pragma unroll
        for (int r = 0; r < 8; ++r) dot8x2(acc2[r], w[r], xv);
    }

    // Whole-row slot of up to 4 rows of K = KS * 2048 (or fewer) columns:
    // thread ct loads its chunk of each piece of each row (4 * KS loads),
    // releases the slot, then accumulates rows into acc[0..3].
    template <int KS>
    __device__ __forceinline__ void mv_rows4(const Ctx &c, int32_t nrows, int32_t nch,
                                             const float (&xr)[kMvResident][8], uint64_t *acc) {
        const uint32_t s = wait_slot(c);
        const uint4 *base = reinterpret_cast<const uint4 *>(c.ring + (size_t)s * slot_bytes);
        uint4 w[4 * KS];
#pragma unroll
        for (int q = 0; q < 4 * KS; ++q) {
            const int r = q / KS, ch = ct + kComputeThreads * (q % KS);
            w[q] = (r < nrows && ch < nch) ? base[r * nch + ch] : make_uint4(0u, 0u, 0u, 0u);
        }
        release_slot(c, s);
#pragma unroll
        for (int q = 0; q < 4 * KS; ++q) dot8x2(acc[q / KS], w[q], xr[q % KS]);
    }

    // Whole-row slot of up to 8 rows of at most 2048 columns.
    __device__ __forceinline__ void mv_rows8(const Ctx &c, int32_t nrows, int32_t nch, const float (&xv)[8],
                                             uint64_t (&acc2)[8]) {
        const uint32_t s = wait_slot(c);
        const uint4 *base = reinterpret_cast<const uint4 *>(c.ring + (size_t)s * slot_bytes) + ct;
        uint4 w[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) w[r] = (r < nrows && ct < nch) ? base[r * nch] : make_uint4(0u, 0u, 0u, 0u);
        release_slot(c, s);
#pragma unroll
        for (int r = 0; r < 8; ++r) dot8x2(acc2[r], w[r], xv);
    }

    // Slot of 4 gate rows then 4 up rows (at most 2048 columns), n of each live.
    __device__ __forceinline__ void mv_rows8_gu(const Ctx &c, int32_t n, int32_t nch, const float (&xv)[8],
                                                uint64_t (&acc2)[8]) {
        const uint32_t s = wait_slot(c);
        const uint4 *base = reinterpret_cast<const uint4 *>(c.ring + (size_t)s * slot_bytes) + ct;
        uint4 w[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) w[r] = ((r & 3) < n && ct < nch) ? base[r * nch] : make_uint4(0u, 0u, 0u, 0u);
        release_slot(c, s);
#pragma unroll
        for (int r = 0; r < 8; ++r) dot8x2(acc2[r], w[r], xv);
    }

    // Both pieces of a two-piece row group at once: 16 loads in flight, then
    // 16 rows x pieces of paired FMAs (more independent work per warp).
    __device__ __forceinline__ void mv_group2(const Ctx &c, int32_t pw8a, int32_t pw8b, int32_t R,
                                              const float (&xa)[8], const float (&xb)[8], uint64_t (&acc2)[8]) {
        const uint32_t sa = wait_slot(c);
        const uint4 *ba = reinterpret_cast<const uint4 *>(c.ring + (size_t)sa * slot_bytes) + ct;
        uint4 wa[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) wa[r] = (ct < pw8a && r < R) ? ba[r * pw8a] : make_uint4(0u, 0u, 0u, 0u);
        release_slot(c, sa);
        const uint32_t sb = wait_slot(c);
        const uint4 *bb = reinterpret_cast<const uint4 *>(c.ring + (size_t)sb * slot_bytes) + ct;
        uint4 wb[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) wb[r] = (ct < pw8b && r < R) ? bb[r * pw8b] : make_uint4(0u, 0u, 0u, 0u);
        release_slot(c, sb);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            dot8x2(acc2[r], wa[r], xa);
            dot8x2(acc2[r], wb[r], xb);
        }
    }

    __device__ void run_matvec(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const int op = t.op;
        const MvGeom g = p.mv[op];
        const int32_t nchunk = g.K / 8;
        const LayerW &lw = p.layers[t.layer];
        const int32_t token = p.tokens[0];
        const bool has_resid = (op == OP_O || op == OP_DOWN);
        const int32_t nrows = t.a1 - t.a0;
        const bool resid_in_smem = has_resid && nrows <= kMaxResid;
        // residual rows of this task: loaded now into registers, stored to
        // shared memory just before the barrier that precedes their first use
        // (so that no warp waits for them at the task's start)
        static_assert(kMaxResid % kComputeThreads == 0, "residual rows per thread");
        float rv[kMaxResid / kComputeThreads];
        bool resid_stored = !resid_in_smem;
        if (resid_in_smem) {
#pragma unroll
            for (int k = 0; k < kMaxResid / kComputeThreads; ++k) {
                const int32_t i = ct + k * kComputeThreads;
                rv[k] = i >= nrows ? 0.f
                                   : ((op == OP_O && t.layer == 0)
                                          ? __uint_as_float((uint32_t)p.embed[(int64_t)token * p.H + t.a0 + i] << 16)
                                          : __ldcg(p.x + t.a0 + i));
            }
        }

        const uint16_t *emb_row = (op == OP_QKV && t.layer == 0) ? p.embed + (int64_t)token * p.H : nullptr;
        const float *xin = (op == OP_O) ? p.attn_out : (op == OP_DOWN ? p.hbuf : p.x);
        const uint16_t *gain =
            op == OP_QKV ? lw.attn_norm : (op == OP_GU ? lw.mlp_norm : (op == OP_LM ? p.final_norm : nullptr));
        const bool resident = g.ksplit <= kMvResident;
        float xr[kMvResident][8];
        uint4 gr[kMvResident];  // RMSNorm gains of the resident chunks, loaded with the input
        float ss = 0.f;
        if (resident || gain != nullptr) {
#pragma unroll
            for (int j = 0; j < kMvResident; ++j)
                load_piece(p, xin, emb_row, nullptr, 1.f, nchunk, j < g.ksplit ? j : 1 << 20, xr[j]);
            if (resident && gain != nullptr) {
#pragma unroll
                for (int j = 0; j < kMvResident; ++j) {
                    const int32_t ch = ct + kComputeThreads * j;
                    gr[j] = ch < nchunk ? __ldg(reinterpret_cast<const uint4 *>(gain) + ch) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int j = 0; j < kMvResident; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(xr[j][e], xr[j][e], ss);
        }
        if (gain != nullptr) {
            // the rest of a streamed input, for the sum of squares only: four
            // pieces' loads in flight at a time (a streamed input without a
            // norm, the down projection's, skips this pass)
            for (int j = kMvResident; j < g.ksplit; j += 4) {
                float v[4][8];
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    load_piece(p, xin, emb_row, nullptr, 1.f, nchunk, j + a < g.ksplit ? j + a : 1 << 20, v[a]);
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(v[a][e], v[a][e], ss);
            }
        }
        float rn = 1.f;
        if (gain != nullptr) {
            // RMSNorm: r = 1/sqrt(mean(x^2) + eps), x-hat = g * x * r
            ss = warp_sum(ss);
            if (lane == 0) c.sc->rms_part[wc] = ss;
            compute_bar();
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kComputeWarps; ++w) tot += c.sc->rms_part[w];
            rn = rsqrtf(tot / (float)g.K + p.eps);
            compute_bar();  // rms_part is reused by the next task
            if (resident) {
#pragma unroll
                for (int j = 0; j < kMvResident; ++j) {
                    const int32_t ch = ct + kComputeThreads * j;
                    if (ch < nchunk) {
                        const uint4 gv = gr[j];
                        xr[j][0] *= rn * bf16_lo(gv.x); xr[j][1] *= rn * bf16_hi(gv.x);
                        xr[j][2] *= rn * bf16_lo(gv.y); xr[j][3] *= rn * bf16_hi(gv.y);
                        xr[j][4] *= rn * bf16_lo(gv.z); xr[j][5] *= rn * bf16_hi(gv.z);
                        xr[j][6] *= rn * bf16_lo(gv.w); xr[j][7] *= rn * bf16_hi(gv.w);
                    }
                }
            }
        }
        const int lq = lane >> 2;  // row this lane holds after the reduce-scatter
        // group geometry and outputs in registers (the ring's inline asm would
        // otherwise force re-reads of the parameter block every slot)
        const int32_t qb1 = p.nq * p.d, qb2 = qb1 + p.nkv * p.d, qb3 = p.qkv_rows;
        float *const out_qkv = p.qkv, *const out_x = p.x, *const out_h = p.hbuf, *const out_logits = p.logits;
        const uint16_t *const embed_row = p.embed + (int64_t)token * p.H;
        int32_t pg = 0;  // row groups waiting in mv_part
        unsigned long long best = 0ull;  // fused greedy pick: this thread's best packed logit
        // a group's 8 row sums, reduced over the warp: lane l ends with value
        // l/4; this warp's totals wait in shared memory, so the warps never
        // meet per group (they drift apart by up to the ring's depth)
        auto park = [&](const uint64_t (&acc2)[8], int32_t grow, int32_t gn) {
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = sum_x2(acc2[r]);
            const float v = warp_reduce8(acc, lane);
            if ((lane & 3) == 0) c.sc->mv_part[pg][lq][wc] = v;
            if (ct == 0) {
                c.sc->mv_grow[pg] = grow;
                c.sc->mv_gn[pg] = gn;
            }
            ++pg;
        };
        // every warp's totals of the waiting groups are in: finish them
        auto flush = [&](bool more) {
            if (!resid_stored) {
#pragma unroll
                for (int k = 0; k < kMaxResid / kComputeThreads; ++k) {
                    const int32_t i = ct + k * kComputeThreads;
                    if (i < nrows) c.sc->resid[i] = rv[k];
                }
                resid_stored = true;
            }
            compute_bar();
            mv_finish(c, t, g, pg, resid_in_smem, out_qkv, out_x, out_h, out_logits, embed_row, best);
            pg = 0;
            if (more) compute_bar();  // the buffer is refilled
        };
        if (!resident) {
            // Inputs longer than kMvResident pieces stream from L2.  Up to
            // kMvSuper row groups go through the pieces together (the
            // producer's order), so each piece is loaded once for all of them,
            // one piece (that is, up to kMvSuper slots) ahead of its use.
            float xc[8], xn[8];
            load_piece(p, xin, emb_row, gain, rn, nchunk, 0, xc);
            for (int32_t row = t.a0; row < t.a1;) {
                int32_t gr[kMvSuper], gn[kMvSuper];
                int32_t r = row;
#pragma unroll
                for (int gi = 0; gi < kMvSuper; ++gi) {
                    int32_t n = 0;
                    if (r < t.a1) {
                        n = min(g.rpp, t.a1 - r);
                        if (op == OP_QKV) n = min(n, (r < qb1 ? qb1 : (r < qb2 ? qb2 : qb3)) - r);
                    }
                    gr[gi] = r;
                    gn[gi] = n;
                    r += n;
                }
                uint64_t acc2[kMvSuper][8];
#pragma unroll
                for (int gi = 0; gi < kMvSuper; ++gi)
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc2[gi][q] = 0ull;
                for (int ks = 0; ks < g.ksplit; ++ks) {
                    // the next piece (piece 0 after the last: the next super-group's first)
                    load_piece(p, xin, emb_row, gain, rn, nchunk, ks + 1 < g.ksplit ? ks + 1 : 0, xn);
                    const int32_t pw8 = min(g.kc, g.K - ks * g.kc) >> 3;
#pragma unroll
                    for (int gi = 0; gi < kMvSuper; ++gi)
                        if (gn[gi] > 0) mv_slot(c, pw8, gn[gi] * g.row_mult, xc, acc2[gi]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) xc[e] = xn[e];
                }
#pragma unroll
                for (int gi = 0; gi < kMvSuper; ++gi)
                    if (gn[gi] > 0) park(acc2[gi], gr[gi], gn[gi]);
                row = r;
                if (pg + kMvSuper > kPartGroups || row >= t.a1) flush(row < t.a1);
            }
        } else {
            for (int32_t row = t.a0; row < t.a1;) {
                int32_t n = min(g.rpp, t.a1 - row);
                if (op == OP_QKV) n = min(n, (row < qb1 ? qb1 : (row < qb2 ? qb2 : qb3)) - row);
                const int32_t R = n * g.row_mult;
                uint64_t acc2[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) acc2[r] = 0ull;
                if (g.rps == 8) {
                    // 8 rows of one matrix, or 4 gate rows (acc 0..3) + 4 up rows (acc 4..7)
                    if (g.row_mult == 2) mv_rows8_gu(c, n, nchunk, xr[0], acc2);
                    else mv_rows8(c, n, nchunk, xr[0], acc2);
                } else if (g.rps == 4) {
                    // acc rows 0..3: first slot; 4..7: the up rows (gate/up) or rows 4..7
                    const int32_t na = (g.row_mult == 2) ? n : min(n, 4), nb = (g.row_mult == 2) ? n : n - 4;
                    if (g.ksplit == 2) {
                        mv_rows4<2>(c, na, nchunk, xr, &acc2[0]);
                        if (nb > 0) mv_rows4<2>(c, nb, nchunk, xr, &acc2[4]);
                    } else {
                        mv_rows4<1>(c, na, nchunk, xr, &acc2[0]);
                        if (nb > 0) mv_rows4<1>(c, nb, nchunk, xr, &acc2[4]);
                    }
                } else if (g.ksplit == 2) {
                    mv_group2(c, g.kc >> 3, (g.K - g.kc) >> 3, R, xr[0], xr[1], acc2);
                } else {
                    mv_slot(c, g.K >> 3, R, xr[0], acc2);
                }
                park(acc2, row, n);
                row += n;
                if (pg == kPartGroups || row >= t.a1) flush(row < t.a1);
            }
        }
        if (op == OP_LM && p.greedy) {
            // fused greedy pick: this CTA's best (logit, row), then one 64-bit
            // max per CTA; the last CTA out writes the token
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
                best = other > best ? other : best;
            }
            if (lane == 0) c.sc->amax_part[wc] = best;
            compute_bar();
            if (ct == 0) {
                for (int w = 1; w < kComputeWarps; ++w) best = c.sc->amax_part[w] > best ? c.sc->amax_part[w] : best;
                if (best != 0ull)
                    atomicMax(reinterpret_cast<unsigned long long *>(p.ctl + p.cl.amax_idx), best);
            }
        }
    }

    // Output rows of the pg waiting groups, one (group, row) per thread: the
    // sum over the warps' totals and the fused epilogue (residual add,
    // SiLU(gate) * up, or the raw value).
    __device__ __forceinline__ void mv_finish(const Ctx &c, const Task &t, const MvGeom &g, int32_t pg,
                                              bool resid_in_smem, float *out_qkv, float *out_x, float *out_h,
                                              float *out_logits, const uint16_t *embed_row,
                                              unsigned long long &best) const {
        const int op = t.op;
        for (int32_t i = ct; i < pg * 8; i += kComputeThreads) {
            const int32_t gi = i >> 3, ri = i & 7;
            const int32_t n = c.sc->mv_gn[gi];
            if (ri >= n) continue;
            const float4 *pv = reinterpret_cast<const float4 *>(&c.sc->mv_part[gi][ri][0]);
            const float4 a = pv[0], b = pv[1];
            const float tot = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
            const int32_t orow = c.sc->mv_grow[gi] + ri;
            switch (op) {
                case OP_QKV: out_qkv[orow] = tot; break;
                case OP_GU: {
                    const int up = (g.rps > 0) ? 4 : n;  // where the group's up rows sit
                    const float4 *pu = reinterpret_cast<const float4 *>(&c.sc->mv_part[gi][up + ri][0]);
                    const float4 ua = pu[0], ub = pu[1];
                    const float tot2 = ((ua.x + ua.y) + (ua.z + ua.w)) + ((ub.x + ub.y) + (ub.z + ub.w));
                    out_h[orow] = tot / (1.f + expf(-tot)) * tot2;
                    break;
                }
                case OP_O:
                case OP_DOWN: {
                    const float xo = resid_in_smem ? c.sc->resid[orow - t.a0]
                                                   : ((op == OP_O && t.layer == 0)
                                                          ? __uint_as_float((uint32_t)embed_row[orow] << 16)
                                                          : __ldcg(out_x + orow));
                    out_x[orow] = xo + tot;
                    break;
                }
                default: {
                    out_logits[orow] = tot;
                    const unsigned long long w = pack_logit(tot, orow);
                    best = w > best ? w : best;
                    break;
                }
            }
        }
    }

    // ------------------------------------------ batched path: projections
    // Units [a0, a1) of the operator, cut by row tile into segments.  The MMA
    // warp issues the MMAs of each segment into one of two TMEM accumulator
    // buffers (mma_role); the eight compute warps read them back and run the
    // fused epilogue, two warps per TMEM lane quarter (warp id mod 4), each
    // of the pair on alternate 16-column chunks.
    __device__ void run_gemm(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const TcGeom g = p.tcg[t.op];
        const int mats = (t.op == OP_GU) ? 2 : 1;
        const int32_t t0 = t.a0 / g.kchunks, t1 = (t.a1 - 1) / g.kchunks;
        epilogue(c, t, g, mats, t0, t1);
        consumed += (uint32_t)((t.a1 - t.a0) * mats);
        aconsumed += (uint32_t)(t.a1 - t.a0);
        seg += (uint32_t)(t1 - t0 + 1);
    }

    // The MMA warp's share of a projection task (one thread): issue its
    // segments, advance the ring counters, record its waits in the trace.
    __device__ bool mma_task(const Ctx &c, const Task &t, uint64_t *tr) {
        const KParams &p = *c.p;
        const TcGeom g = p.tcg[t.op];
        const int mats = (t.op == OP_GU) ? 2 : 1;
        const int32_t t0 = t.a0 / g.kchunks, t1 = (t.a1 - 1) / g.kchunks;
        const uint32_t c0 = consumed, a0 = aconsumed;
        const bool ok = mma_issuer(c, t, g, mats, t0, t1);
        consumed = c0 + (uint32_t)((t.a1 - t.a0) * mats);
        aconsumed = a0 + (uint32_t)(t.a1 - t.a0);
        seg += (uint32_t)(t1 - t0 + 1);
        if (tr) {
            tr[3] = full_wait_ns;
            tr[6] = act_wait_ns;
            tr[7] = acc_wait_ns;
            full_wait_ns = act_wait_ns = acc_wait_ns = 0;
        }
        return ok;
    }

    // One thread.  Slot indices and phase bits advance by increments, and the
    // operand descriptors are the ring bases' plus the slot offset (the
    // start-address field is the low 14 bits, address / 16): a unit costs
    // its waits, four or eight MMAs and the commits, no division.
    __device__ bool mma_issuer(const Ctx &c, const Task &t, const TcGeom &g, int mats, int32_t t0, int32_t t1) {
        const KParams &p = *c.p;
        SmemCtl *sc = c.sc;
        const uint32_t nas = (uint32_t)p.num_aslots;
        uint32_t wi = consumed % ns, wph = (consumed / ns) & 1u;
        uint32_t ai = aconsumed % nas, aph = (aconsumed / nas) & 1u;
        const uint64_t wdesc0 = umma_desc_sw128(smem_u32(c.ring)), adesc0 = umma_desc_sw128(smem_u32(c.aring));
        const uint32_t wstep = slot_bytes >> 4, astep = (uint32_t)p.aslot_bytes >> 4;
        const uint32_t idesc = p.idesc, mstride = 2u * (uint32_t)p.npad;
        const int sub = p.tc_sub;
        // descriptor offset of sub-tile j: weights 128 x 64 bf16 = 16 KB apart,
        // activations the slot's share
        const uint32_t wsub = (uint32_t)(kTcTileM * kTcTileK * 2) >> 4, asub = ((uint32_t)p.aslot_bytes / sub) >> 4;
        uint32_t sg = seg;
        for (int32_t tile = t0; tile <= t1; ++tile, ++sg) {
            const int32_t klo = (tile == t0) ? t.a0 % g.kchunks : 0;
            const int32_t khi = (tile == t1) ? (t.a1 - 1) % g.kchunks + 1 : g.kchunks;
            const uint32_t ab = sg & 1u, use = sg >> 1;
            uint64_t t0 = tracing ? globaltimer_ns() : 0;
            if (!wait_mbar(c, &sc->acc_empty[ab], (use & 1u) ^ 1u, SITE_ACC_WAIT)) return false;
            if (tracing) acc_wait_ns += globaltimer_ns() - t0;
            tc_fence_after();
            const uint32_t dcol = sc->tmem_base + ab * 2u * mstride;
            for (int32_t k = klo; k < khi; ++k) {
                uint32_t ws[2] = {0u, 0u};
                if (tracing) t0 = globaltimer_ns();
                for (int m = 0; m < mats; ++m) {
                    ws[m] = wi;
                    if (!wait_mbar(c, &sc->full[wi], wph, SITE_FULL_WAIT)) return false;
                    if (++wi == ns) {
                        wi = 0;
                        wph ^= 1u;
                    }
                }
                if (tracing) {
                    const uint64_t t1 = globaltimer_ns();
                    full_wait_ns += t1 - t0;
                    t0 = t1;
                }
                const uint32_t as = ai;
                if (!wait_mbar(c, &sc->afull[as], aph, SITE_FULL_WAIT)) return false;
                if (++ai == nas) {
                    ai = 0;
                    aph ^= 1u;
                }
                if (tracing) act_wait_ns += globaltimer_ns() - t0;
                tc_fence_after();
                const uint64_t ad = adesc0 + (uint64_t)(as * astep);
                for (int m = 0; m < mats; ++m) {
                    const uint64_t wd = wdesc0 + (uint64_t)(ws[m] * wstep);
                    for (int j = 0; j < sub; ++j)
#pragma unroll
                        for (int kk = 0; kk < kTcTileK / 16; ++kk)  // K = 16 bf16 = 32 bytes = 2 descriptor units
                            umma_bf16(dcol + (uint32_t)m * mstride, wd + j * wsub + 2u * kk, ad + j * asub + 2u * kk,
                                      idesc, (k > klo || j > 0 || kk > 0) ? 1u : 0u);
                }
                for (int m = 0; m < mats; ++m) umma_commit(&sc->empty[ws[m]]);
                umma_commit(&sc->aempty[as]);
            }
            umma_commit(&sc->acc_full[ab]);
        }
        consumed += (uint32_t)((t.a1 - t.a0) * mats);
        aconsumed += (uint32_t)(t.a1 - t.a0);
        return true;
    }

    // Epilogue warps: for each segment, wait for its accumulator, publish or
    // gather the partial sums of a shared row tile, and finish the tile.
    __device__ void epilogue(const Ctx &c, const Task &t, const TcGeom &g, int mats, int32_t t0, int32_t t1) {
        const KParams &p = *c.p;
        SmemCtl *sc = c.sc;
        const int op = t.op;
        const int q4 = (wc + 2) & 3;  // TMEM lane quarter of this warp (its warp id mod 4)
        const int r = q4 * 32 + lane; // row of the tile held by this thread
        const int et = ct;            // 0..255
        const int cfirst = 16 * (wc >> 2);  // this warp's first 16-column chunk; it takes every other one
        if (op == OP_QKV || op == OP_GU || op == OP_LM) {
            // RMSNorm scale of each sequence from the producers' per-tile sums of x^2
            for (int b = et; b < p.B; b += kEpiThreads) {
                float ssum = 0.f;
                for (int j = 0; j < p.h_tiles; ++j) ssum += __ldcg(p.ssq + (size_t)b * p.h_tiles + j);
                sc->rs[b] = rsqrtf(ssum / (float)p.H + p.eps);
                sc->amax_seq[b] = 0ull;
            }
        }
        epi_bar();
        const int64_t U = g.units, NR = g.nranges;
        const int32_t rc = t.a2;  // this task's range number
        uint32_t sg = seg;
        for (int32_t tile = t0; tile <= t1; ++tile, ++sg) {
            const int32_t klo = (tile == t0) ? t.a0 % g.kchunks : 0;
            const int32_t khi = (tile == t1) ? (t.a1 - 1) % g.kchunks + 1 : g.kchunks;
            const uint32_t ab = sg & 1u, use = sg >> 1;
            wait_mbar(c, &sc->acc_full[ab], use & 1u, SITE_ACC_WAIT);
            tc_fence_after();
            const uint32_t tq = sc->tmem_base + ((uint32_t)(q4 * 32) << 16) + ab * 4u * (uint32_t)p.npad;
            const bool whole = (klo == 0 && khi == g.kchunks);
            int32_t cf = rc, cl = rc;
            bool last = true;
            if (!whole) {
                // several ranges share this row tile: publish this partial sum,
                // the last range to arrive adds them all up in range order
                const int64_t tu0 = (int64_t)tile * g.kchunks;
                cf = range_of(tu0, U, NR);
                cl = range_of(tu0 + g.kchunks - 1, U, NR);
                float *mine = part_ptr(p, rc, tile, g);
                for (int m = 0; m < mats; ++m)
                    for (int c0 = cfirst; c0 < p.npad; c0 += 32) {
                        float v[16];
                        tmem_ld_split16(tq + (uint32_t)(m * 2 * p.npad + c0), p.npad, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) __stcg(mine + ((size_t)m * p.npad + c0 + i) * kTcTileM + r, v[i]);
                    }
                // the barrier, then one acq_rel atomic (cumulative release) publishes every thread's partial
                epi_bar();
                if (et == 0) {
                    uint32_t n_contrib = 0;  // non-empty ranges meeting this tile
                    for (int32_t cc = cf; cc <= cl; ++cc) n_contrib += range_nonempty(cc, U, NR) ? 1u : 0u;
                    uint32_t *ctr = p.tile_ctr + g.ctr_off + tile;
                    const uint32_t old = atom_acq_rel_gpu_add(ctr, 1u);
                    const bool l = (old + 1u == n_contrib);
                    if (l) *ctr = 0u;  // every range of this tile has arrived; ready for the next use
                    sc->ep_last = l ? 1u : 0u;
                }
                epi_bar();
                last = sc->ep_last != 0u;
            }
            if (last) {
                if (mats == 2) finish_tile<2>(c, t, g, tile, r, tq, whole, cf, cl, rc);
                else finish_tile<1>(c, t, g, tile, r, tq, whole, cf, cl, rc);
            }
            tc_fence_before();
            epi_bar();
            if (et == 0) mbar_arrive(&sc->acc_empty[ab]);
        }
        if (op == OP_LM && p.greedy) {
            // fused greedy pick: this CTA's best (logit, row) of every sequence,
            // one 64-bit max per sequence; the last CTA out writes the tokens
            for (int b = et; b < p.B; b += kEpiThreads)
                if (sc->amax_seq[b] != 0ull)
                    atomicMax(reinterpret_cast<unsigned long long *>(p.ctl + p.cl.amax_idx) + b, sc->amax_seq[b]);
        }
    }

    // Partial-sum slot [2][npad][128] of range rc for row tile `tile`: slot 0
    // when the tile is the range's first, else slot 1 (its last).
    __device__ static float *part_ptr(const KParams &p, int32_t rc, int32_t tile, const TcGeom &g) {
        const int64_t first_tile = range_start(rc, g.units, g.nranges) / g.kchunks;
        const int sidx = (first_tile == tile) ? 0 : 1;
        return p.part + ((size_t)rc * 2 + sidx) * 2 * (size_t)p.npad * kTcTileM;
    }

    // MATS (1, or 2 for gate/up) is a template argument: the gate/up tile's
    // second accumulator is not held live in the single-matrix epilogues.
    template <int MATS>
    __device__ void finish_tile(const Ctx &c, const Task &t, const TcGeom &g, int32_t tile, int r, uint32_t tq,
                                bool whole, int32_t cf, int32_t cl, int32_t rc) {
        constexpr int mats = MATS;
        const KParams &p = *c.p;
        SmemCtl *sc = c.sc;
        const int op = t.op;
        const int q4 = (wc + 2) & 3;
        const int et = ct;
        // where this thread's row goes
        int32_t orow = tile * kTcTileM + r, obase = 0, olim = g.rows;
        if (op == OP_QKV) {
            const int32_t qr = p.nq * p.d, kr = p.nkv * p.d;
            if (tile < g.tiles_q) {
                olim = qr;
            } else if (tile < g.tiles_q + g.tiles_k) {
                orow = (tile - g.tiles_q) * kTcTileM + r;
                obase = qr;
                olim = kr;
            } else {
                orow = (tile - g.tiles_q - g.tiles_k) * kTcTileM + r;
                obase = qr + kr;
                olim = kr;
            }
        }
        const bool row_ok = orow < olim;
        float gain = 0.f;
        if ((op == OP_O || op == OP_DOWN) && row_ok) {
            const uint16_t *gv = (op == OP_O) ? p.layers[t.layer].mlp_norm
                                              : (t.layer + 1 < p.L ? p.layers[t.layer + 1].attn_norm : p.final_norm);
            gain = __uint_as_float((uint32_t)gv[orow] << 16);
        }
        const bool resid = (op == OP_O || op == OP_DOWN);
        for (int c0 = 16 * (wc >> 2); c0 < p.npad; c0 += 32) {
            // the residual stream's values are read before the partial sums,
            // all independent loads, so that one round trip covers them
            float xo[16];
            if (resid) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    xo[i] = (c0 + i < p.B && row_ok) ? __ldcg(p.x + (size_t)(c0 + i) * p.H + orow) : 0.f;
            }
            float v[mats][16];
#pragma unroll
            for (int m = 0; m < mats; ++m) {
                if (whole) {
                    tmem_ld_split16(tq + (uint32_t)(m * 2 * p.npad + c0), p.npad, v[m]);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[m][i] = 0.f;
                    // kFix contributing ranges' partial sums are loaded at once, then
                    // added in range order (the same sums, fewer round trips; more
                    // than two at once spills registers)
                    constexpr int kFix = 2;
                    for (int32_t cg = cf; cg <= cl; cg += kFix) {
                        float w[kFix][16];
#pragma unroll
                        for (int j = 0; j < kFix; ++j) {
                            const int32_t cc = cg + j;
                            if (cc == rc) {
                                tmem_ld_split16(tq + (uint32_t)(m * 2 * p.npad + c0), p.npad, w[j]);
                            } else if (cc <= cl && range_nonempty(cc, g.units, g.nranges)) {
                                const float *src = part_ptr(p, cc, tile, g) + ((size_t)m * p.npad + c0) * kTcTileM + r;
#pragma unroll
                                for (int i = 0; i < 16; ++i) w[j][i] = __ldcg(src + (size_t)i * kTcTileM);
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i) w[j][i] = 0.f;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < kFix; ++j)
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[m][i] += w[j][i];
                    }
                }
            }
            float sq[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                sq[i] = 0.f;
                const int b = c0 + i;
                if (b >= p.B || !row_ok) continue;
                switch (op) {
                    case OP_QKV: p.qkv[(size_t)b * p.qkv_rows + obase + orow] = sc->rs[b] * v[0][i]; break;
                    case OP_O:
                    case OP_DOWN: {
                        const size_t xi = (size_t)b * p.H + orow;
                        const float xn = xo[i] + v[0][i];
                        p.x[xi] = xn;
                        store_split(p.xa, p.H, p.npad, b, orow, gain * xn);
                        sq[i] = xn * xn;
                        break;
                    }
                    case OP_GU: {
                        const float gg = sc->rs[b] * v[0][i], uu = sc->rs[b] * v[mats - 1][i];
                        store_split(p.h_a, p.I, p.npad, b, orow, gg / (1.f + expf(-gg)) * uu);
                        break;
                    }
                    default: p.logits[(size_t)b * p.V + orow] = sc->rs[b] * v[0][i]; break;
                }
            }
            if (resid) {
                // per-warp sums of x^2 for the 16 sequences of this chunk
                const float s16 = warp_reduce16(sq, lane);
                if ((lane & 1) == 0) sc->ssq_red[q4][c0 + ((lane >> 1) & 15)] = s16;
            }
            if (op == OP_LM && p.greedy) {
                // this warp's best (logit, row) of each of the chunk's 16 sequences
                unsigned long long key[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    key[i] = (c0 + i < p.B && row_ok) ? pack_logit(sc->rs[c0 + i] * v[0][i], orow) : 0ull;
                const unsigned long long k16 = warp_max16_u64(key, lane);
                if ((lane & 1) == 0 && k16 != 0ull) atomicMax(&sc->amax_seq[c0 + ((lane >> 1) & 15)], k16);
            }
        }
        if (op == OP_O || op == OP_DOWN) {
            epi_bar();
            for (int b = et; b < p.B; b += kEpiThreads)
                p.ssq[(size_t)b * p.h_tiles + tile] =
                    sc->ssq_red[0][b] + sc->ssq_red[1][b] + sc->ssq_red[2][b] + sc->ssq_red[3][b];
        }
    }

    // ------------------------------------------ batched path: embedding
    // Items [a0, a1) = (sequence, 128-row tile of H): x = embed[token],
    // xa = bf16(attn_norm_0 * x), and the tile's sum of x^2.
    __device__ void run_embed(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const uint16_t *gain = p.layers[0].attn_norm;
        for (int32_t it = t.a0; it < t.a1; ++it) {
            const int32_t b = it / p.h_tiles, j = it % p.h_tiles;
            const int32_t tok = p.tokens[(int64_t)b * p.tok_stride];
            float sq = 0.f;
            const int32_t row = j * kTcTileM + ct;
            if (ct < kTcTileM && row < p.H) {
                const float e = __uint_as_float((uint32_t)p.embed[(int64_t)tok * p.H + row] << 16);
                const size_t xi = (size_t)b * p.H + row;
                p.x[xi] = e;
                store_split(p.xa, p.H, p.npad, b, row, __uint_as_float((uint32_t)gain[row] << 16) * e);
                sq = e * e;
            }
            sq = warp_sum(sq);
            if (lane == 0) c.sc->rms_part[wc] = sq;
            compute_bar();
            if (ct == 0) {
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < kComputeWarps; ++w) tot += c.sc->rms_part[w];
                p.ssq[(size_t)b * p.h_tiles + j] = tot;
            }
            compute_bar();
        }
    }

    // ------------------------------------------- kv-append graphs: OP_KVA
    // Items [a0, a1) = (batch row, kv head): RoPE on the row's new k, both
    // rounded to bf16 and stored at its position in the paged cache, where
    // the attention tasks of every row then read it (by TMA: the stores are
    // fenced for the async proxy).
    __device__ void run_kva(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        const int half = p.d / 2;
        for (int32_t it = t.a0; it < t.a1; ++it) {
            const int32_t b = it / p.nkv, kvh = it % p.nkv;
            const int32_t pos = p.positions[(int64_t)b * p.pos_stride];
            const int32_t page = p.page_table[(int64_t)b * p.pt_stride + pos / p.page_size];
            const float *kh = p.qkv + (int64_t)b * p.qkv_rows + (int64_t)p.nq * p.d + (int64_t)kvh * p.d;
            const float *vh = kh + (int64_t)p.nkv * p.d;
            const int64_t off = kv_offset(p, t.layer, page, kvh, pos % p.page_size);
            if (ct < half) {
                const float ka = __ldcg(kh + ct), kb = __ldcg(kh + ct + half);
                const float2 cs = p.rope[(int64_t)pos * half + ct];
                p.k_pool[off + ct] = f32_to_bf16_bits(ka * cs.x - kb * cs.y);
                p.k_pool[off + ct + half] = f32_to_bf16_bits(ka * cs.y + kb * cs.x);
            }
            if (ct < p.d) p.v_pool[off + ct] = f32_to_bf16_bits(__ldcg(vh + ct));
        }
        fence_proxy_async_global();  // read next by the attention tasks' TMA
    }

    // ---------------------------------------------------- attention task
    // One (sequence, kv head, context split) task.  The G query heads of the
    // kv head are split into bf16 high and low parts (2G MMA columns), so the
    // bf16 tensor-core products keep about 16 significant bits of q and of
    // the softmax weights.  Per 64-token block of the cache:
    //   scores  S^T[tok][2G] = K[tok][d] Q^T     (warps 0..3, 16 tokens each)
    //   online softmax per head                  (warp g for head g)
    //   O^T[d][2G] += V^T[d][tok] P^T[tok][2G]   (warp w for rows 16w..16w+15)
    // with mma.sync m16n8k16 (bf16 in, fp32 accumulate) on K/V tiles that the
    // producer laid out 128-byte swizzled, so every ldmatrix is conflict-free.

    // Shared-memory address of element e of token `tok` (0..63) of the K
    // (kv = 0) or V (kv = 1) tile of a block held in slots sb0 (tokens
    // [0, ts)) and sb1 (tokens [ts, 64)); ts = 1 << ts_log2.  Shifts and a
    // select only: no local-memory array, no integer division.
    __device__ static __forceinline__ uint32_t kv_elem(uint32_t sb0, uint32_t sb1, int ts_log2, int halves, int kv,
                                                       int tok, int e) {
        const int ti = tok & ((1 << ts_log2) - 1), h = e >> 6, ch = (e & 63) >> 3;
        return ((tok >> ts_log2) ? sb1 : sb0) +
               (uint32_t)((((kv * halves + h) * 128) << ts_log2) + ti * 128 + ((ch ^ (ti & 7)) << 4) + (e & 7) * 2);
    }

    // The same for the tokens of an attention step held in up to four slots
    // (token tok of the step lies in slot tok >> ts_log2).
    __device__ static __forceinline__ uint32_t kv_elem4(uint32_t sb0, uint32_t sb1, uint32_t sb2, uint32_t sb3,
                                                        int ts_log2, int halves, int kv, int tok, int e) {
        const int sl = tok >> ts_log2;
        const uint32_t lo = (sl & 1) ? sb1 : sb0, hi = (sl & 1) ? sb3 : sb2;
        return kv_elem((sl & 2) ? hi : lo, 0u, ts_log2, halves, kv, tok & ((1 << ts_log2) - 1), e);
    }

    // Long context splits (G <= 4 query heads per kv head, at least four
    // blocks): each step holds two 64-token blocks, and warp w takes tokens
    // 16w..16w+15 of it through the whole computation in registers, with no
    // barrier inside the step.  Scores S^T = K Q^T (m16n8k16, split-bf16
    // queries as 2G columns); an online softmax over the warp's own tokens
    // (running max and sum per head); the weights split into bf16 high and
    // low parts, moved from the scores' accumulator layout to the B-operand
    // layout by an 8x8 transpose (movmatrix); O^T[d][2G] += V^T P^T over all
    // d rows.  After the last step the eight warps' (m, l, O) are merged in a
    // three-round tree through shared memory, and the result is left where
    // the per-block path leaves it: oacc (warp w: rows 16w.. of d, high
    // columns; low columns 0) and att_m, att_l.
    __device__ void attend_warps(const Ctx &c, const AttnRange &r, int layer, int G, int nks, int halves, int nsl,
                                 int ts_log2, uint32_t qb, float (&oacc)[2][4]) {
        SmemCtl *sc = c.sc;
        const int tr = lane >> 2, cq = lane & 3;
        const int partner = (G >= 2) ? G / 2 : 0;   // lane distance to the low-part column (G <= 4)
        const bool head_lane = (G == 1) ? cq == 0 : cq < G / 2;
        const bool pad_lane = (G == 2 && cq >= 2) || (G == 1 && cq != 0);
        float o2[8][4];  // O^T rows 16 mt + tr (+8), columns 2 cq (+1): this warp's tokens
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) o2[mt][i] = 0.f;
        float wm[2] = {-INFINITY, -INFINITY}, wl[2] = {0.f, 0.f};  // head lanes: heads 2cq, 2cq+1
        // This warp's 16 tokens of a step lie in one slot (the step's slot
        // wsl); the ldmatrix addresses of its K and V fragments within that
        // slot are the same every step, so they are computed once here:
        // kof[ks] (K rows 16 wc + lane % 16, columns 16 ks + 8 (lane / 16))
        // and vof[mt] (V rows 16 wc + 8 (q / 2) + lane % 8, columns 16 mt +
        // 8 (q % 2), q = lane / 8).
        const int wsl = (16 * wc) >> ts_log2;
        uint32_t kof[8], vof[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            kof[j] = kv_elem(0u, 0u, ts_log2, halves, 0, (16 * wc + (lane & 15)) & ((1 << ts_log2) - 1),
                             j * 16 + (lane >> 4) * 8);
            const int q = lane >> 3;
            vof[j] = kv_elem(0u, 0u, ts_log2, halves, 1, (16 * wc + (q >> 1) * 8 + (lane & 7)) & ((1 << ts_log2) - 1),
                             16 * j + (q & 1) * 8);
        }
        // the queries' B-operand fragments are the same every step: held in registers
        uint32_t qfr[8][2];
        {
            const uint32_t qlane = qb + (uint32_t)(((lane & 7) * kQhlStride + ((lane >> 3) & 1) * 8) * 2);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                if (ks < nks) ldsm_x2(qfr[ks], qlane + (uint32_t)(ks * 32));
        }
        // the softmax runs in base 2: scores times log2(e), so that each
        // weight is one exp2; the running maxima are converted back at the end
        constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
        const uint64_t tb0 = tracing ? globaltimer_ns() : 0;
        for (int32_t blk = r.blo; blk < r.bhi; blk += 2) {
            const int NB = (blk + 1 < r.bhi) ? 2 : 1;
            const int nslots = NB * nsl;
            const int32_t tok0 = blk * kAttnBlock;
            if (wc < 4 * NB) {
                // only this warp's slot: every slot of the step is released
                // together after the barrier below, so no warp runs a lap ahead
                const uint32_t sbw = smem_u32(c.ring + (size_t)wait_slot_at(c, consumed + (uint32_t)wsl) * slot_bytes);
                // even and odd column slices accumulate separately: two
                // independent chains of dependent MMAs instead of one
                float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sodd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    if (ks < nks) {
                        uint32_t a[4];
                        ldsm_x4(a, sbw + kof[ks]);
                        mma_bf16_16816((ks & 1) ? sodd : sacc, a, qfr[ks]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) sacc[i] += sodd[i];
                // scores of (token row, head) in the head lanes; -inf past the context
                float sv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = sacc[i];
                    if (G == 1) v = (i & 1) ? 0.f : sacc[i] + sacc[i + 1];
                    else v += __shfl_xor_sync(0xFFFFFFFFu, v, partner);
                    const int tok = 16 * wc + tr + (i >> 1) * 8;
                    sv[i] = (tok0 + tok < r.ctx) ? v * kLog2e : -INFINITY;
                }
                // the step's maximum per head over this warp's 16 tokens
                float mx[2] = {fmaxf(sv[0], sv[2]), fmaxf(sv[1], sv[3])};
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xFFFFFFFFu, mx[j], o));
                float alpha[2], nm[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    nm[j] = fmaxf(wm[j], mx[j]);
                    alpha[j] = (nm[j] == -INFINITY || wm[j] == -INFINITY) ? (nm[j] == -INFINITY ? 1.f : 0.f)
                                                                         : exp2f(wm[j] - nm[j]);
                }
                float pv[4], ps[2] = {0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    pv[i] = (sv[i] == -INFINITY) ? 0.f : exp2f(sv[i] - nm[i & 1]);
                    ps[i & 1] += pv[i];
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) ps[j] += __shfl_xor_sync(0xFFFFFFFFu, ps[j], o);
                    wl[j] = wl[j] * alpha[j] + ps[j];
                    wm[j] = nm[j];
                }
                // rescale this warp's O: each lane's columns belong to its own
                // heads (high parts) or to its partner's (low parts)
                float ca0 = alpha[0], ca1 = alpha[1];
                if (G >= 2) {
                    const float r0 = __shfl_xor_sync(0xFFFFFFFFu, alpha[0], partner);
                    const float r1 = __shfl_xor_sync(0xFFFFFFFFu, alpha[1], partner);
                    if (!head_lane) {
                        ca0 = r0;
                        ca1 = r1;
                    }
                } else {
                    ca1 = alpha[0];  // G = 1: columns 0 and 1 are head 0's high and low parts
                }
                // (most steps leave every head's maximum where it was)
                if (__any_sync(0xFFFFFFFFu, ca0 != 1.f || ca1 != 1.f)) {
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        o2[mt][0] *= ca0;
                        o2[mt][1] *= ca1;
                        o2[mt][2] *= ca0;
                        o2[mt][3] *= ca1;
                    }
                }
                // the weights as the B operand P^T[16 tokens][2G columns]:
                // high parts in the head lanes' columns, low parts in their
                // partners', bf16 pairs transposed 8x8
                float hi[4], lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    hi[i] = __uint_as_float((uint32_t)f32_to_bf16_bits(pv[i]) << 16);
                    lo[i] = pv[i] - hi[i];
                }
                float val[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (G == 1) {
                        val[i] = (i & 1) ? lo[i - 1] : hi[i];
                    } else {
                        const float lr = __shfl_xor_sync(0xFFFFFFFFu, lo[i], partner);
                        val[i] = head_lane ? hi[i] : lr;
                    }
                    if (pad_lane) val[i] = 0.f;
                }
                const uint32_t r0 = (uint32_t)f32_to_bf16_bits(val[0]) | ((uint32_t)f32_to_bf16_bits(val[1]) << 16);
                const uint32_t r1 = (uint32_t)f32_to_bf16_bits(val[2]) | ((uint32_t)f32_to_bf16_bits(val[3]) << 16);
                const uint32_t b[2] = {movmatrix_trans(r0), movmatrix_trans(r1)};
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    if (mt < nks) {
                        uint32_t a[4];
                        ldsm_x4_trans(a, sbw + vof[mt]);
                        mma_bf16_16816(o2[mt], a, b);
                    }
                }
            }
            compute_bar();  // the step's slots are free
            if (ct == 0) {
                const uint32_t na = c.p->tc ? 1u : (uint32_t)kComputeWarps;
                for (int j = 0; j < nslots; ++j) mbar_arrive_n(&sc->empty[(consumed + (uint32_t)j) % ns], na);
            }
            consumed += (uint32_t)nslots;
        }
        // the head lanes' per-head O: high plus low column
        float oh[8][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float v = o2[mt][i];
                if (G == 1) v = (i & 1) ? 0.f : o2[mt][i] + o2[mt][i + 1];
                else v += __shfl_xor_sync(0xFFFFFFFFu, v, partner);
                oh[mt][i] = v;
            }
        // tree merge of the warps' (m, l, O) through shared memory: warps
        // 4..7 into 0..3, 2..3 into 0..1, 1 into 0
        float *mo = &sc->at.s_s[0][0];       // [4][kMaxHeadDim][4] partial O
        float *mm = mo + 4 * kMaxHeadDim * 4;  // [4][4] running max
        float *ml = mm + 16;                   // [4][4] sum
        const int dd = nks * 16;
        for (int half = 4; half >= 1; half >>= 1) {
            if (wc >= half && wc < 2 * half && head_lane) {
                const int slot = wc - half;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int h = (G == 1) ? 0 : 2 * cq + (i & 1);
                        if (mt < nks && (G != 1 || (i & 1) == 0))
                            mo[(slot * kMaxHeadDim + 16 * mt + tr + (i >> 1) * 8) * 4 + h] = oh[mt][i];
                    }
                if (tr == 0) {
                    const int h0 = (G == 1) ? 0 : 2 * cq;
                    mm[slot * 4 + h0] = wm[0];
                    ml[slot * 4 + h0] = wl[0];
                    if (G != 1) {
                        mm[slot * 4 + h0 + 1] = wm[1];
                        ml[slot * 4 + h0 + 1] = wl[1];
                    }
                }
            }
            compute_bar();
            if (wc < half && head_lane) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (G == 1 && j == 1) continue;
                    const int h = (G == 1) ? 0 : 2 * cq + j;
                    const float mb = mm[wc * 4 + h], lb = ml[wc * 4 + h];
                    const float M = fmaxf(wm[j], mb);
                    const float wa = (wm[j] == -INFINITY) ? 0.f : exp2f(wm[j] - M);
                    const float wb = (mb == -INFINITY) ? 0.f : exp2f(mb - M);
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                        for (int i = j; i < 4; i += 2)
                            if (mt < nks)
                                oh[mt][i] = oh[mt][i] * wa +
                                            mo[(wc * kMaxHeadDim + 16 * mt + tr + (i >> 1) * 8) * 4 + h] * wb;
                    wl[j] = wl[j] * wa + lb * wb;
                    wm[j] = M;
                }
            }
            compute_bar();
        }
        // warp 0 holds the split's result: per-head O to shared memory, then
        // every warp takes its rows of d in the per-block path's layout
        if (wc == 0 && head_lane) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int h = (G == 1) ? 0 : 2 * cq + (i & 1);
                    if (mt < nks && (G != 1 || (i & 1) == 0)) mo[(16 * mt + tr + (i >> 1) * 8) * 4 + h] = oh[mt][i];
                }
            if (tr == 0) {  // running maxima back in natural units
                const int h0 = (G == 1) ? 0 : 2 * cq;
                sc->att_m[h0] = wm[0] * kLn2;
                sc->att_l[h0] = wl[0];
                if (G != 1) {
                    sc->att_m[h0 + 1] = wm[1] * kLn2;
                    sc->att_l[h0 + 1] = wl[1];
                }
            }
        }
        compute_bar();
        if (wc < nks) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int col = 2 * cq + (i & 1);
                const int e = 16 * wc + tr + (i >> 1) * 8;
                oacc[0][i] = (col < G && e < dd) ? mo[e * 4 + col] : 0.f;
                oacc[1][i] = 0.f;
            }
        }
        compute_bar();  // the merge buffer (the scores' scratch) is free
        if (tracing) act_wait_ns += globaltimer_ns() - tb0;
    }

    __device__ void run_attn(const Ctx &c, const Task &t) {
        const KParams &p = *c.p;
        SmemCtl *sc = c.sc;
        const int d = p.d, half = d / 2, halves = d / 64, nks = d / 16;
        const int G = p.nq / p.nkv, NT = (2 * G + 7) / 8;
        const int b = t.a0, kvh = t.a1, S = t.a3;
        const AttnRange r = attn_range(p, t);
        // a split with no cached block and without the new token neither
        // computes nor takes part in the merge (short contexts leave most
        // splits empty)
        if (r.blo == r.bhi && !r.has_new) return;
        const float *qkv = p.qkv + (int64_t)b * p.qkv_rows;
        const float2 *rope = p.rope + (int64_t)r.pos * half;
        const float scale = rsqrtf((float)d);
        const int ts = p.attn_ts, nsl = kAttnBlock / ts, ts_log2 = (ts == 64) ? 6 : 5;

        // Every load of the setup (queries, RoPE factors, the new token's k
        // and v, its page) is issued before any is used: one round trip.
        // Thread ct: query pairs (idx, idx + d/2) for idx = ct, ct + 256
        // (G d/2 <= 512), the k pair (ct, ct + d/2), v element ct (d <= 128).
        const float *kh = qkv + (int64_t)p.nq * d + (int64_t)kvh * d;
        const float *vh = qkv + (int64_t)(p.nq + p.nkv) * d + (int64_t)kvh * d;
        float qa[2] = {0.f, 0.f}, qb2[2] = {0.f, 0.f}, ka = 0.f, kb = 0.f, vv = 0.f;
        float2 qcs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, kcs = make_float2(0.f, 0.f);
        int32_t new_page = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int idx = ct + kComputeThreads * k;
            if (idx < G * half) {
                const float *qh = qkv + (int64_t)(kvh * G + idx / half) * d + idx % half;
                qa[k] = __ldcg(qh);
                qb2[k] = __ldcg(qh + half);
                qcs[k] = rope[idx % half];
            }
        }
        if (r.has_new) {
            if (ct < half) {
                ka = __ldcg(kh + ct);
                kb = __ldcg(kh + ct + half);
                kcs = rope[ct];
            }
            if (ct < d) vv = __ldcg(vh + ct);
            new_page = p.page_table[(int64_t)b * p.pt_stride + r.pos / p.page_size];
        }
        // RoPE'd, pre-scaled queries of the G heads sharing this kv head, in
        // fp32 and split into bf16 high / low parts (rows G..2G-1 the low parts)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int idx = ct + kComputeThreads * k;
            if (idx >= G * half) continue;
            const int g = idx / half, i = idx % half;
            const float a = qa[k], bb = qb2[k];
            const float2 cs = qcs[k];
            const float q0 = (a * cs.x - bb * cs.y) * scale, q1 = (a * cs.y + bb * cs.x) * scale;
            sc->at.q_s[g][i] = q0;
            sc->at.q_s[g][i + half] = q1;
            const uint16_t h0 = f32_to_bf16_bits(q0), h1 = f32_to_bf16_bits(q1);
            sc->at.q_hl[g][i] = h0;
            sc->at.q_hl[g][i + half] = h1;
            sc->at.q_hl[G + g][i] = f32_to_bf16_bits(q0 - __uint_as_float((uint32_t)h0 << 16));
            sc->at.q_hl[G + g][i + half] = f32_to_bf16_bits(q1 - __uint_as_float((uint32_t)h1 << 16));
        }
        // MMA columns past 2G stay zero
        for (int idx = ct; idx < (8 * NT - 2 * G) * kQhlStride; idx += kComputeThreads)
            sc->at.q_hl[2 * G + idx / kQhlStride][idx % kQhlStride] = 0;
        for (int idx = ct; idx < (8 * NT - 2 * G) * kPhlStride; idx += kComputeThreads)
            sc->at.p_hl[2 * G + idx / kPhlStride][idx % kPhlStride] = 0;
        if (r.has_new) {
            // K/V of the new token: RoPE on k, round to bf16, append to the cache
            const int64_t off = kv_offset(p, t.layer, new_page, kvh, r.pos % p.page_size);
            if (ct < half) {
                const uint16_t k0 = f32_to_bf16_bits(ka * kcs.x - kb * kcs.y);
                const uint16_t k1 = f32_to_bf16_bits(ka * kcs.y + kb * kcs.x);
                sc->knew[ct] = k0;
                sc->knew[ct + half] = k1;
                p.k_pool[off + ct] = k0;
                p.k_pool[off + ct + half] = k1;
            }
            if (ct < d) {
                const uint16_t v = f32_to_bf16_bits(vv);
                sc->vnew[ct] = v;
                p.v_pool[off + ct] = v;
            }
        }
        if (ct < G) {
            sc->att_m[ct] = -INFINITY;
            sc->att_l[ct] = 0.f;
        }
        compute_bar();

        const uint32_t qb = smem_u32(&sc->at.q_hl[0][0]);  // B operand (Q^T) of the score MMAs
        // hi/lo column pairing of the MMA C fragment: column n holds the high
        // part of head n (n < G) or the low part of head n - G
        const int tr = lane >> 2, cq = lane & 3;
        const int partner = (G == 8) ? 0 : (G >= 2 ? G / 2 : 0);  // lane distance to the low-part column
        const bool head_lane = (G == 8) || (G == 1 ? cq == 0 : cq < G / 2);
        float oacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};

        // One step: NB (1 or 2) consecutive 64-token blocks, held in NB * nsl
        // ring slots.  Two blocks per step halve the barriers per token and
        // put all 8 warps on the scores (16 tokens each).
        auto attend = [&](auto nb_const, int32_t blk) {
            constexpr int NB = decltype(nb_const)::value;
            const int nslots = NB * nsl;
            const uint64_t tb0 = tracing ? globaltimer_ns() : 0;
            const uint32_t sid0 = wait_slot_at(c, consumed);
            const uint32_t sid1 = (nslots > 1) ? wait_slot_at(c, consumed + 1u) : sid0;
            const uint32_t sid2 = (nslots > 2) ? wait_slot_at(c, consumed + 2u) : sid0;
            const uint32_t sid3 = (nslots > 3) ? wait_slot_at(c, consumed + 3u) : sid0;
            const uint32_t sb0 = smem_u32(c.ring + (size_t)sid0 * slot_bytes);
            const uint32_t sb1 = smem_u32(c.ring + (size_t)sid1 * slot_bytes);
            const uint32_t sb2 = smem_u32(c.ring + (size_t)sid2 * slot_bytes);
            const uint32_t sb3 = smem_u32(c.ring + (size_t)sid3 * slot_bytes);
            const int32_t tok0 = blk * kAttnBlock;
            // scores of tokens 16 wc .. 16 wc + 15 of the step
            if (wc < 4 * NB) {
                float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    if (ks < nks) {
                        uint32_t a[4], qf[2];
                        ldsm_x4(a, kv_elem4(sb0, sb1, sb2, sb3, ts_log2, halves, 0, 16 * wc + (lane & 15),
                                            ks * 16 + (lane >> 4) * 8));
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            if (nt < NT) {
                                ldsm_x2(qf, qb + (uint32_t)((((lane & 7) + 8 * nt) * kQhlStride + ks * 16 +
                                                             ((lane >> 3) & 1) * 8) * 2));
                                mma_bf16_16816(sacc[nt], a, qf);
                            }
                        }
                    }
                }
                // sum the high and low parts, mask tokens past the cached context
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = sacc[0][i];
                    if (G == 8) v += sacc[1][i];
                    else if (G == 1) v = (i & 1) ? 0.f : sacc[0][i] + sacc[0][i + 1];
                    else v += __shfl_xor_sync(0xFFFFFFFFu, v, partner);
                    const int tok = 16 * wc + tr + (i >> 1) * 8;
                    const int head = (G == 1) ? 0 : 2 * cq + (i & 1);
                    const bool live = head_lane && (G != 1 || (i & 1) == 0);
                    if (live) sc->at.s_s[head][tok] = (tok0 + tok < r.ctx) ? v : -INFINITY;
                }
            }
            compute_bar();
            const uint64_t tb1 = tracing ? globaltimer_ns() : 0;
            // online softmax, warp g for head g: weights as bf16 high / low parts
            if (wc < G) {
                const int g = wc;
                float sv[2 * NB], pv[2 * NB];
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < 2 * NB; ++j) {
                    sv[j] = sc->at.s_s[g][lane + 32 * j];
                    mx = fmaxf(mx, sv[j]);
                }
                const float m_old = sc->att_m[g];
                const float m_new = fmaxf(m_old, warp_max(mx));
                float psum = 0.f;
#pragma unroll
                for (int j = 0; j < 2 * NB; ++j) {
                    pv[j] = (sv[j] == -INFINITY) ? 0.f : expf(sv[j] - m_new);
                    psum += pv[j];
                    const uint16_t h = f32_to_bf16_bits(pv[j]);
                    sc->at.p_hl[g][lane + 32 * j] = h;
                    sc->at.p_hl[G + g][lane + 32 * j] = f32_to_bf16_bits(pv[j] - __uint_as_float((uint32_t)h << 16));
                }
                const float sum = warp_sum(psum);
                if (lane == 0) {
                    const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
                    sc->att_alpha[g] = alpha;
                    sc->att_l[g] = sc->att_l[g] * alpha + sum;
                    sc->att_m[g] = m_new;
                }
            }
            compute_bar();
            const uint64_t tb2 = tracing ? globaltimer_ns() : 0;
            // O^T rows 16 wc .. 16 wc + 15: rescale, then add V^T P^T
            if (wc < nks) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int col = nt * 8 + 2 * cq + (i & 1);
                        if (nt < NT && col < 2 * G) oacc[nt][i] *= sc->att_alpha[col % G];
                    }
                const uint32_t pb = smem_u32(&sc->at.p_hl[0][0]);
#pragma unroll
                for (int k2 = 0; k2 < NB * kAttnBlock / 16; ++k2) {
                    uint32_t a[4];
                    const int q = lane >> 3;
                    ldsm_x4_trans(a, kv_elem4(sb0, sb1, sb2, sb3, ts_log2, halves, 1,
                                              k2 * 16 + (q >> 1) * 8 + (lane & 7), 16 * wc + (q & 1) * 8));
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        if (nt < NT) {
                            uint32_t bq[2];
                            ldsm_x2(bq, pb + (uint32_t)((((lane & 7) + 8 * nt) * kPhlStride + k2 * 16 +
                                                         ((lane >> 3) & 1) * 8) * 2));
                            mma_bf16_16816(oacc[nt], a, bq);
                        }
                    }
                }
            }
            compute_bar();  // the step's slots, scores and weights are free
            if (ct == 0) {
                const uint32_t na = p.tc ? 1u : (uint32_t)kComputeWarps;
                mbar_arrive_n(&sc->empty[sid0], na);
                if (nslots > 1) mbar_arrive_n(&sc->empty[sid1], na);
                if (nslots > 2) mbar_arrive_n(&sc->empty[sid2], na);
                if (nslots > 3) mbar_arrive_n(&sc->empty[sid3], na);
            }
            consumed += (uint32_t)nslots;
            if (tracing) {
                act_wait_ns += tb1 - tb0;            // slot waits + scores
                acc_wait_ns += globaltimer_ns() - tb2;  // value sums
            }
        };
        if (G <= 4 && r.bhi - r.blo >= 4 && ns >= (uint32_t)(2 * nsl)) {
            // long splits: every warp runs its own tokens end to end
            attend_warps(c, r, t.layer, G, nks, halves, nsl, ts_log2, qb, oacc);
        } else {
            // pairs of blocks while the ring can hold both at once, then the rest
            int32_t blk = r.blo;
            if (ns >= (uint32_t)(2 * nsl))
                for (; blk + 1 < r.bhi; blk += 2) attend(std::integral_constant<int, 2>{}, blk);
            for (; blk < r.bhi; ++blk) attend(std::integral_constant<int, 1>{}, blk);
        }
        if (r.has_new) {
            // the new token, from shared memory: one more online-softmax step
            if (wc < G) {
                const int g = wc;
                float sdot = 0.f;
                for (int e = lane; e < d; e += 32) sdot = fmaf(sc->at.q_s[g][e], __uint_as_float((uint32_t)sc->knew[e] << 16), sdot);
                sdot = warp_sum(sdot);
                if (lane == 0) {
                    const float m_old = sc->att_m[g], m_new = fmaxf(m_old, sdot);
                    const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
                    const float pn = expf(sdot - m_new);
                    sc->att_alpha[g] = alpha;
                    sc->att_pnew[g] = pn;
                    sc->att_l[g] = sc->att_l[g] * alpha + pn;
                    sc->att_m[g] = m_new;
                }
            }
            compute_bar();
            if (wc < nks) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int col = nt * 8 + 2 * cq + (i & 1);
                        if (nt < NT && col < 2 * G) {
                            const int e = 16 * wc + tr + (i >> 1) * 8;
                            const float vn = __uint_as_float((uint32_t)sc->vnew[e] << 16);
                            oacc[nt][i] = oacc[nt][i] * sc->att_alpha[col % G] + (col < G ? sc->att_pnew[col] * vn : 0.f);
                        }
                    }
            }
            compute_bar();
        }
        if (r.n_live == 1) {
            // The only split with work (at most one cached block, or one
            // split in all): normalise in registers and write the heads'
            // outputs; no partial, no split counter, no merge.  The result is
            // the merge's for one split, bit for bit (its weight is exp(0)).
            if (wc < nks) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = oacc[0][i];
                    if (G == 8) v += oacc[1][i];
                    else if (G == 1) v = (i & 1) ? 0.f : oacc[0][i] + oacc[0][i + 1];
                    else v += __shfl_xor_sync(0xFFFFFFFFu, v, partner);
                    const int e = 16 * wc + tr + (i >> 1) * 8;
                    const int head = (G == 1) ? 0 : 2 * cq + (i & 1);
                    const bool live = head_lane && (G != 1 || (i & 1) == 0);
                    if (live) {
                        const float o = v * (1.f / sc->att_l[head]);
                        const int64_t col = (int64_t)(kvh * G + head) * d + e;
                        if (p.tc) store_split(p.attn_a, p.nq * d, p.npad, b, col, o);
                        else p.attn_out[(int64_t)b * p.nq * d + col] = o;
                    }
                }
            }
            if (p.tc) fence_proxy_async_global();  // read next by the O projection's TMA
            compute_bar();
            if (ct == 0 && p.only_op < 0 && t.signal_ev != kNoEvent && !local_abort(c))
                red_release_gpu_add(p.ctl + t.signal_ev, 1u);  // cumulative: every output written before the barrier
            return;
        }
        // partial result of this split: unnormalised o (high + low columns), running max, sum
        // partial sums of pair (b, kvh) at a stride of the plan's largest split count
        const int64_t pidx = (((int64_t)b * p.nkv + kvh) * p.attn_splits + t.a2) * G;
        if (wc < nks) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float v = oacc[0][i];
                if (G == 8) v += oacc[1][i];
                else if (G == 1) v = (i & 1) ? 0.f : oacc[0][i] + oacc[0][i + 1];
                else v += __shfl_xor_sync(0xFFFFFFFFu, v, partner);
                const int e = 16 * wc + tr + (i >> 1) * 8;
                const int head = (G == 1) ? 0 : 2 * cq + (i & 1);
                const bool live = head_lane && (G != 1 || (i & 1) == 0);
                if (live) p.attn_part[(pidx + head) * (d + 2) + e] = v;
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
            const uint32_t old = atom_acq_rel_gpu_add(done, 1u);  // releases the partials written before the barrier
            sc->last_flag = (old + 1u == (uint32_t)r.n_live) ? 1u : 0u;  // empty splits never arrive
        }
        compute_bar();
        if (sc->last_flag) {
            // last split of this (sequence, kv head) to finish: merge the
            // partials of the live splits.  Split weights exp(m_j - M) and 1/L
            // first (warp g, lane j: the running max and sum of live split j,
            // one round trip), then every thread sums its output pairs over
            // the splits, eight loads in flight at a time.
            if (ct == 0) *done = 0u;  // nothing else touches it in this launch
            const int64_t pbase = ((int64_t)b * p.nkv + kvh) * p.attn_splits * G;
            if (wc < G) {
                const int g = wc;
                float M = -INFINITY;
                for (int j0 = 0; j0 < r.n_live; j0 += 32) {
                    const int j = j0 + lane;
                    float ms = -INFINITY, ls = 0.f;
                    if (j < r.n_live) {
                        const float *src = p.attn_part + (pbase + (int64_t)live_split(r.ctx, j, S) * G + g) * (d + 2);
                        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(src + d));
                        ms = ml.x;
                        ls = ml.y;
                        sc->merge_w[j][g] = ms;  // m_j for now, the weight below
                        sc->merge_l[j][g] = ls;
                    }
                    M = fmaxf(M, warp_max(ms));
                }
                float Ls = 0.f;
                for (int j = lane; j < r.n_live; j += 32) {
                    const float ms = sc->merge_w[j][g];
                    const float w = (ms == -INFINITY) ? 0.f : expf(ms - M);
                    sc->merge_w[j][g] = w;
                    Ls = fmaf(sc->merge_l[j][g], w, Ls);
                }
                Ls = warp_sum(Ls);
                if (lane == 0) sc->att_inv_l[g] = 1.f / Ls;
            }
            compute_bar();
            const int npairs = G * half;  // output pairs: (head, even column)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (ct + kComputeThreads * k < npairs) {
                    const int pr = ct + kComputeThreads * k;
                    const int g = pr / half, e = (pr % half) * 2;
                    const float *src = p.attn_part + (pbase + g) * (d + 2) + e;
                    const int64_t sstride = (int64_t)G * (d + 2);
                    float o0 = 0.f, o1 = 0.f;
                    constexpr int kChunk = 8;
                    for (int j0 = 0; j0 < r.n_live; j0 += kChunk) {
                        float2 v[kChunk];
#pragma unroll
                        for (int j = 0; j < kChunk; ++j)
                            v[j] = (j0 + j < r.n_live)
                                       ? __ldcg(reinterpret_cast<const float2 *>(src + live_split(r.ctx, j0 + j, S) * sstride))
                                       : make_float2(0.f, 0.f);
#pragma unroll
                        for (int j = 0; j < kChunk; ++j) {
                            const float w = (j0 + j < r.n_live) ? sc->merge_w[j0 + j][g] : 0.f;
                            o0 = fmaf(v[j].x, w, o0);
                            o1 = fmaf(v[j].y, w, o1);
                        }
                    }
                    const float il = sc->att_inv_l[g];
                    const int64_t oi = (int64_t)b * p.nq * d + (int64_t)(kvh * G + g) * d + e;
                    if (p.tc) {
                        // split-bf16 operand of the O projection's tensor-core tiles
                        const int64_t col = (int64_t)(kvh * G + g) * d + e;
                        store_split(p.attn_a, p.nq * d, p.npad, b, col, o0 * il);
                        store_split(p.attn_a, p.nq * d, p.npad, b, col + 1, o1 * il);
                    } else {
                        *reinterpret_cast<float2 *>(p.attn_out + oi) = make_float2(o0 * il, o1 * il);
                    }
                }
            }
            if (p.tc) fence_proxy_async_global();  // read next by the O projection's TMA
            compute_bar();
            if (ct == 0 && p.only_op < 0 && t.signal_ev != kNoEvent && !local_abort(c))
                red_release_gpu_add(p.ctl + t.signal_ev, 1u);  // cumulative: every row written before the barrier
        }
    }
};

// Wait (bounded) until the scheduler has released queue position i; false
// on the scheduler's abort mark, a local abort or a timeout (recorded).
__device__ bool wait_ready(const Ctx &c, int i) {
    uint32_t r = ld_acquire_cta(&c.sc->ready);
    if (r == kReadyAbort) return false;
    if (r >= (uint32_t)(i + 1)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        r = ld_acquire_cta(&c.sc->ready);
        if (r == kReadyAbort) return false;
        if (r >= (uint32_t)(i + 1)) return true;
        if ((it & 63u) == 0) {
            if (local_abort(c)) return false;
            if (globaltimer_ns() - t0 > 4 * c.p->timeout_ns) {
                record_error(c, 4, SITE_READY_WAIT, i);
                return false;
            }
        }
    }
}

template <bool JIT>
__device__ void compute_role(const Ctx &c, const Task *q, int nt) {
    const KParams &p = *c.p;
    Consumer cs;
    cs.ns = (uint32_t)p.num_slots;
    cs.slot_bytes = (uint32_t)p.slot_bytes;
    cs.tcm = p.tc != 0;
    cs.ct = threadIdx.x - 64;
    cs.wc = cs.ct >> 5;
    cs.lane = threadIdx.x & 31;
    cs.tracing = p.trace != nullptr && !JIT && cs.ct == 0;
    for (int i = 0;; ++i) {
        Task t;
        if (JIT) {
            // every compute thread reads the claimed task, then they meet (so
            // that the slot is free again only once all hold it); the end of
            // the claims is seen alike by all of them
            const bool got = jit_task(c, i, &t, nullptr);
            if (compute_bar_or(local_abort(c))) return;
            if (!got) break;
            if (cs.ct == 0) st_release_cta(&c.sc->jcomp, (uint32_t)(i + 1));
        } else {
            if (i >= nt) break;
            t = q[i];
        }
        if (!task_active(p, t)) continue;
        wait_ready(c, i);  // the scheduler releases task i (an abort is seen at the barrier below)
        if (compute_bar_or(local_abort(c))) return;  // every compute warp takes the same branch
        uint64_t *tr = cs.tracing ? trace_slot(p, i) : nullptr;
        if (tr) tr[1] = globaltimer_ns();
        if (t.op == OP_ATTN) cs.run_attn(c, t);
        else if (t.op == OP_EMBED) cs.run_embed(c, t);
        else if (t.op == OP_KVA) cs.run_kva(c, t);
        else if (p.tc) cs.run_gemm(c, t);
        else cs.run_matvec(c, t);
        // batched path: outputs are read by other CTAs' TMA (async proxy)
        if (p.tc) fence_proxy_async_global();
        const bool aborted = compute_bar_or(local_abort(c));  // every output row of the task is written
        if (tr) {
            tr[2] = globaltimer_ns();
            if (!(p.tc && is_proj(t.op))) {  // a projection's waits are the MMA warp's
                tr[3] = cs.full_wait_ns;
                tr[6] = cs.act_wait_ns;
                tr[7] = cs.acc_wait_ns;
            }
            cs.full_wait_ns = cs.act_wait_ns = cs.acc_wait_ns = 0;
        }
        if (aborted) return;
        // a gpu-scope release is cumulative: it also publishes the other
        // compute warps' output rows, ordered before it by the barrier above
        if (t.op != OP_ATTN && p.only_op < 0 && t.signal_ev != kNoEvent && cs.ct == 0)
            red_release_gpu_add(p.ctl + t.signal_ev, 1u);
    }
}

// JIT: dynamic dispatch (tasks claimed at run time); otherwise every CTA
// walks its static queue.
// ------------------------------------------------------------- MMA warp
// Batched path: one thread walks the same task sequence as the compute warps
// and issues every projection's tcgen05 MMAs; for an attention task it only
// counts the ring slots the compute warps consume, so that its slot and
// phase arithmetic stays in step with theirs.  A projection waits for its
// release by the scheduler first: its dependencies include this CTA's
// earlier tasks, so by then every slot counted for them has been consumed
// and the ring's phases (one parity bit per slot) are the ones counted.
// Without that wait the warp would reach a weight slot's barrier laps ahead
// of the attention tasks still cycling the ring.
template <bool JIT>
__device__ void mma_role(const Ctx &c, const Task *q, int nt) {
    const KParams &p = *c.p;
    if (!p.tc || (threadIdx.x & 31) != 0) return;
    Consumer ms;
    ms.ns = (uint32_t)p.num_slots;
    ms.slot_bytes = (uint32_t)p.slot_bytes;
    ms.tcm = true;
    ms.ct = -1;
    ms.wc = -1;
    ms.lane = 0;
    ms.tracing = p.trace != nullptr && !JIT;
    for (int i = 0;; ++i) {
        Task t;
        if (JIT) {
            if (!jit_task(c, i, &t, &c.sc->jmma)) break;
        } else {
            if (i >= nt) break;
            t = q[i];
        }
        if (!task_active(p, t)) continue;
        if (is_proj(t.op)) {
            if (!wait_ready(c, i)) break;
            if (!ms.mma_task(c, t, ms.tracing ? trace_slot(p, i) : nullptr)) break;
        } else if (t.op == OP_ATTN) {
            const AttnRange r = attn_range(p, t);
            if (r.blo < r.bhi) ms.consumed += (uint32_t)((r.bhi - r.blo) * (kAttnBlock / p.attn_ts));
        }
    }
}

template <bool JIT>
__global__ void __launch_bounds__(kThreads, 1) megakernel(const __grid_constant__ KParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SmemCtl *sc = reinterpret_cast<SmemCtl *>(smem_raw);
    const uint32_t ctl_end = smem_u32(smem_raw) + (uint32_t)sizeof(SmemCtl);
    uint8_t *ring = smem_raw + (((ctl_end + 1023u) & ~1023u) - smem_u32(smem_raw));
    Ctx c{&p, sc, ring, ring + (size_t)p.num_slots * p.slot_bytes, (int)blockIdx.x};
    const Task *q = JIT ? p.tasks : p.tasks + p.queue_off[blockIdx.x];
    const int nt = JIT ? 0 : p.queue_off[blockIdx.x + 1] - p.queue_off[blockIdx.x];
    const int warp = threadIdx.x >> 5;
    constexpr int kWarpMma = 2 + kComputeWarps;  // batched path: TMEM owner and MMA issuer (the last warp)

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.num_slots; ++s) {
            mbar_init(&sc->full[s], 1);
            mbar_init(&sc->empty[s], p.tc ? 1 : kComputeWarps);
        }
        if (p.tc) {
            for (int s = 0; s < p.num_aslots; ++s) {
                mbar_init(&sc->afull[s], 1);
                mbar_init(&sc->aempty[s], 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&sc->acc_full[i], 1);
                mbar_init(&sc->acc_empty[i], 1);
            }
            mbar_init(&sc->mma_done, 1);
        }
        sc->ready = 0;
        sc->abort = global_abort(p) ? 1u : 0u;  // a recorded error stays sticky
        sc->last_flag = 0;
        sc->jclaimed = sc->jdone = sc->jprod = sc->jcomp = sc->jmma = 0;
        fence_mbar_init();
    }
    if (p.tc && warp == kWarpMma) {
        tmem_alloc(&sc->tmem_base, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
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
                const int32_t pg = p.page_table[(int64_t)b * p.pt_stride + j];
                if (pg < 0 || pg >= p.num_pages) {
                    record_error(c, 5, SITE_PAGE, pg);
                    break;
                }
            }
        }
    }
    __syncthreads();
    if (!local_abort(c)) {
        if (warp == kWarpSched) scheduler_role<JIT>(c, q, nt);
        else if (warp == kWarpProd) producer_role<JIT>(c, q, nt);
        else if (warp == kWarpMma) mma_role<JIT>(c, q, nt);
        else compute_role<JIT>(c, q, nt);
    }
    if (p.tc && threadIdx.x == kWarpMma * 32) {
        // no MMA may still be reading shared memory or writing TMEM at exit
        umma_commit(&sc->mma_done);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&sc->mma_done, 0)) {
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                record_error(c, 4, SITE_DRAIN_WAIT, -1);
                break;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (p.tc && warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(sc->tmem_base, p.tmem_cols);
    }
    if (threadIdx.x == 0) {
        // the last CTA out resets the counters for the next launch
        __threadfence();
        uint32_t *ex = p.ctl + p.cl.exit_idx;
        const uint32_t old = atom_acq_rel_gpu_add(ex, 1u);
        if (old == gridDim.x - 1) {
            for (int i = 0; i < p.cl.n_events + p.cl.n_done + p.cl.n_claims; ++i) p.ctl[i] = 0u;
            *ex = 0u;
            if (p.greedy && !p.skip_lm && (p.only_op < 0 || p.only_op == OP_LM) && !global_abort(p)) {
                // fused greedy pick: every CTA's maximum is in
                unsigned long long *am = reinterpret_cast<unsigned long long *>(p.ctl + p.cl.amax_idx);
                for (int b = 0; b < p.B; ++b) {
                    const unsigned long long w = __ldcg(am + b);
                    p.next_tokens[b] = (w == 0ull) ? 0x7FFFFFFF : (int32_t)(0xFFFFFFFFu - (uint32_t)w);
                    p.next_positions[b] += 1;
                    am[b] = 0ull;
                }
            }
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

__global__ void prefill_rows_kernel(const int32_t *src, int32_t n, int32_t p0, int32_t rows, int32_t *tok,
                                    int32_t *pos) {
    const int32_t j = threadIdx.x;
    if (j < rows) {
        const int32_t jj = j < n ? j : n - 1;
        tok[j] = src[jj];
        pos[j] = p0 + jj;
    }
}

template <bool JIT>
const void *kernel_ptr() {
    return reinterpret_cast<const void *>(&megakernel<JIT>);
}

const void *variant_ptr(int variant) { return variant == 1 ? kernel_ptr<true>() : kernel_ptr<false>(); }

}  // namespace

size_t megakernel_smem_bytes(int32_t slot_bytes, int32_t num_slots, int32_t aslot_bytes, int32_t num_aslots) {
    return kRingOffset + (size_t)slot_bytes * num_slots + (size_t)aslot_bytes * num_aslots;
}

int megakernel_variant(int32_t /*max_k*/, bool /*tc*/, bool jit) {
    return jit ? 1 : 0;  // one build per dispatch mode; matvec inputs past 4096 columns stream through L2
}

cudaError_t megakernel_set_smem(int variant, size_t smem) {
    // The dynamic shared-memory limit belongs to the kernel function, so every
    // plan and call in the process shares it: only ever raise it, or a plan
    // made earlier with a larger ring could no longer launch.
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    cudaFuncAttributes a{};
    cudaError_t e = cudaFuncGetAttributes(&a, variant_ptr(variant));
    if (e != cudaSuccess) return e;
    if ((size_t)a.maxDynamicSharedSizeBytes >= smem) return cudaSuccess;
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

namespace mk {

cudaError_t launch_prefill_rows(const int32_t *src, int32_t n, int32_t p0, int32_t rows, int32_t *tok, int32_t *pos,
                                cudaStream_t stream) {
    if (n < 1 || rows < 1 || rows > 1024) return cudaErrorInvalidValue;
    prefill_rows_kernel<<<1, rows, 0, stream>>>(src, n, p0, rows, tok, pos);
    return cudaGetLastError();
}

}  // namespace mk
