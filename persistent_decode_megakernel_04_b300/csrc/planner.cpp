// planner.cpp — host task-graph builder.
//
// Refines the decoder's operator graph into SM-level tasks linked by event
// counters, in the manner of the task graph the MPK compiler emits ("Compilar
// LLM en un MegaKernel…", section "Parte 1. Compilador": each task is a unit
// of work for one SM, events are synchronisation points between tasks, and
// dependencies are tracked at the level of the data actually consumed) and
// of the SM-level tGraph ("MPK: A Compiler and Runtime for Mega-Kernelizing
// Tensor Programs", section 2).
//
// Per layer, in queue order:
//   QKV  : RMSNorm + [Wq;Wk;Wv] rows          waits x ready      signals EV(QKV)
//   ATTN : RoPE + KV append + split attention waits EV(QKV)       last split signals EV(ATTN)
//   O    : split merge + Wo rows + residual    waits EV(ATTN)     signals EV(O)
//   GU   : RMSNorm + gate/up rows + SiLU*mul   waits EV(O)        signals EV(GU)
//   DOWN : Wd rows + residual                  waits EV(GU)       signals EV(DOWN)
// then the LM head (final RMSNorm + W_lm rows) waits the last EV(DOWN).
// Every matvec operator's rows are cut into one contiguous range per worker
// CTA, balanced to within one row; the schedule is fixed ahead of time for a
// (shape, batch) pair, because only the attention length changes between
// steps, and that is resolved on the device from the positions.
#include "planner.h"

#include <algorithm>
#include <cstring>
#include <numeric>
#include <random>

namespace mk {

namespace {

// A row is cut into pieces of kMvPiece columns (one 16-byte chunk per compute
// thread), so piece ks of every row meets the same register-resident input
// chunk in each thread.  A slot holds rpp rows (of each matrix, for gate/up)
// of one piece; at most 8 accumulators per thread.
constexpr int32_t kMvPiece = 2048;

MvGeom make_geom(int32_t K, int32_t rows, int32_t row_mult, int32_t slot_bytes) {
    MvGeom g{};
    g.K = K;
    g.rows = rows;
    g.row_mult = row_mult;
    g.kc = std::min(K, kMvPiece);
    g.ksplit = (K + g.kc - 1) / g.kc;
    if (g.ksplit <= 2 && slot_bytes >= 4 * K * 2) {
        // whole-row slots: one contiguous copy per slot, 4 (or 8 short) rows of one matrix
        // (gate/up at most 2048 columns: 4 gate rows and the matching 4 up rows
        // share a slot, as two contiguous copies; rps = 8 then counts both)
        g.rpp = 8 / row_mult;
        g.rps = (g.ksplit == 1 && slot_bytes >= 8 * K * 2) ? 8 : 4;
    } else {
        g.rpp = std::min(8 / row_mult, slot_bytes / (row_mult * g.kc * 2));
        g.rps = 0;
    }
    return g;
}

}  // namespace

mk_status check_cfg(const mk_model_cfg &c) {
    if (c.n_layers <= 0 || c.hidden <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 ||
        c.ffn_dim <= 0 || c.vocab <= 0 || c.batch <= 0 || c.max_seq <= 0 || c.page_size <= 0)
        return MK_ERR_INVALID;
    if (c.n_q_heads % c.n_kv_heads != 0) return MK_ERR_INVALID;
    if (!(c.rms_eps >= 0.0f) || !(c.rope_theta > 0.0f)) return MK_ERR_INVALID;
    // 16-byte copies need every row length to be a multiple of 8 bf16
    if (c.hidden % 8 || c.ffn_dim % 8 || c.head_dim % 64) return MK_ERR_UNSUPPORTED;
    if (c.n_layers * 6 + 1 >= 0xFFFF) return MK_ERR_UNSUPPORTED;
    const int32_t group = c.n_q_heads / c.n_kv_heads;
    if (group > 8 || (group & (group - 1)) || c.head_dim > 128) return MK_ERR_UNSUPPORTED;
    if (c.page_size % 64) return MK_ERR_UNSUPPORTED;  // attention reads aligned 64-token blocks of a page
    if (c.batch > kTcMaxBatch) return MK_ERR_UNSUPPORTED;  // one tcgen05 N tile holds the whole batch
    return MK_OK;
}

mk_plan_options resolve_options(const mk_model_cfg &cfg, const mk_plan_options *opt, int32_t num_sms) {
    mk_plan_options o;
    std::memset(&o, 0, sizeof(o));
    if (opt) o = *opt;
    if (o.num_ctas <= 0 || o.num_ctas > num_sms) o.num_ctas = num_sms;
    if (o.slot_bytes <= 0) o.slot_bytes = 32768;
    const bool tc = cfg.batch > 1 || o.tensor_cores == 1;
    if (o.num_slots <= 0) o.num_slots = tc ? 0 : 6;  // tensor-core path: as many as shared memory holds
    if (o.timeout_ms <= 0) o.timeout_ms = 2000;
    if (o.attn_splits <= 0) {
        int32_t pairs = cfg.batch * cfg.n_kv_heads;
        o.attn_splits = std::max(1, o.num_ctas / std::max(1, pairs));
    }
    if (o.attn_splits > kMaxSplits) o.attn_splits = kMaxSplits;
    if (o.l2_prefetch_kb < 0) o.l2_prefetch_kb = 0;
    // batch 1: three copies in flight per CTA stream at full bandwidth and
    // keep the queue ahead of this SM's other memory requests (and the
    // release fences, which wait for them) short; measured 1.7% faster than
    // two at the 8B shape, and than four
    if (o.max_inflight <= 0) o.max_inflight = tc ? 0 : 3;
    return o;
}

namespace {

TcGeom make_tc_geom(int32_t K, int32_t rows, int32_t ctr_off, int32_t sub) {
    TcGeom t{};
    t.K = K;
    t.rows = rows;
    t.tiles = (rows + kTcTileM - 1) / kTcTileM;
    t.kchunks = (K + kTcTileK * sub - 1) / (kTcTileK * sub);  // units of sub 64-column sub-tiles
    t.units = t.tiles * t.kchunks;
    t.ctr_off = ctr_off;
    return t;
}

}  // namespace

mk_status build_plan(const mk_model_cfg &cfg, const mk_plan_options &opt, PlanTables *out) {
    mk_status st = check_cfg(cfg);
    if (st != MK_OK) return st;
    const int32_t N = opt.num_ctas;
    const bool tc = cfg.batch > 1 || opt.tensor_cores == 1;
    if (opt.jit < 0 || opt.jit > 16 || (opt.jit > 0 && opt.trace)) return MK_ERR_INVALID;
    if (N <= 0 || opt.slot_bytes < 4096 || opt.slot_bytes % 1024 || opt.attn_splits <= 0 ||
        opt.attn_splits > kMaxSplits || (tc ? (opt.num_slots == 1 || opt.num_slots < 0) : opt.num_slots < 2))
        return MK_ERR_INVALID;
    const int32_t H = cfg.hidden, d = cfg.head_dim, nq = cfg.n_q_heads, nkv = cfg.n_kv_heads;
    const int32_t I = cfg.ffn_dim, V = cfg.vocab, L = cfg.n_layers, B = cfg.batch;
    // Context splits of each (sequence, kv head) pair.  With more pairs than
    // CTAs and one split asked for (the default there), the pairs left over
    // after whole rounds of CTAs are cut into k splits, k (at most 8) chosen
    // to minimise the last round's length: ceil(R k / N) tasks of 1/k of a
    // pair's work plus a fixed cost per task (setup, partial, merge) taken
    // as 0.12 of a pair's.  Batch 64 of 8 kv heads on 148 CTAs: 444 whole
    // pairs, 68 pairs in halves, 3.5 pairs' work on the busiest CTA, not 4.
    const int32_t P = B * nkv;
    std::vector<int32_t> psplit(P, opt.attn_splits);
    if (opt.attn_splits == 1 && P > N && !opt.jit) {
        const int32_t R = P % N;
        if (R > 0) {
            constexpr double kTaskCost = 0.12;
            int32_t best_k = 1;
            double best = 1.0 + kTaskCost;
            for (int32_t k = 2; k <= 8; ++k) {
                const double t = (double)((R * k + N - 1) / N) * (1.0 / k + kTaskCost);
                if (t < best * 0.98) {
                    best = t;
                    best_k = k;
                }
            }
            for (int32_t i = P - R; i < P; ++i) psplit[i] = best_k;
        }
    }
    const int32_t S = *std::max_element(psplit.begin(), psplit.end());  // partial-sum stride per pair

    PlanGeom &g = out->g;
    g = PlanGeom{};
    g.tc = tc;
    g.num_ctas = N;
    g.attn_splits = S;
    if (opt.tc_k_subtiles < 0 || opt.tc_k_subtiles > 2) return MK_ERR_INVALID;
    // two sub-tiles measured faster at batch 8, 32 and 64 (half the MMA
    // warp's waits and commits per weight byte outweigh the shallower ring)
    if (tc) g.tc_sub = opt.tc_k_subtiles > 0 ? opt.tc_k_subtiles : 2;
    g.slot_bytes = tc ? kTcTileM * kTcTileK * 2 * g.tc_sub : opt.slot_bytes;
    g.num_slots = opt.num_slots;
    // KV tokens per ring slot: a 64-token attention block fills 1 or 2 slots
    g.tps = (g.slot_bytes >= 2 * d * 2 * 64) ? 64 : 32;
    if (g.slot_bytes < 2 * d * 2 * 32) return MK_ERR_INVALID;
    const int32_t per = opt.kv_append ? 6 : 5;  // events per layer
    g.kv_append = opt.kv_append != 0;
    g.n_events = per * L + (tc ? 1 : 0);
    g.l2_prefetch_bytes = opt.l2_prefetch_kb * 1024;
    g.max_inflight = opt.max_inflight;
    if (g.tps < 1) return MK_ERR_INVALID;
    if (!tc) {
        g.mv[OP_QKV] = make_geom(H, (nq + 2 * nkv) * d, 1, opt.slot_bytes);
        g.mv[OP_O] = make_geom(nq * d, H, 1, opt.slot_bytes);
        g.mv[OP_GU] = make_geom(H, I, 2, opt.slot_bytes);
        g.mv[OP_DOWN] = make_geom(I, H, 1, opt.slot_bytes);
        g.mv[OP_LM] = make_geom(H, V, 1, opt.slot_bytes);
        for (int op = OP_QKV; op <= OP_LM; ++op)
            if (op != OP_ATTN && g.mv[op].rpp < 1) return MK_ERR_INVALID;  // slot smaller than one row piece
    } else {
        g.npad = (B + 15) / 16 * 16;
        // activation tiles hold 2 * npad rows: the bf16 high parts, then the bf16 low parts
        g.aslot_bytes = 2 * g.npad * kTcTileK * 2 * g.tc_sub;
        // 40 KB of activation slots: one more 32 KB weight slot fits at batch
        // 8 to 32 (measured 1.4-2% faster than 48 KB), batch 64 keeps two
        g.num_aslots = std::max(2, std::min(8, (40 * 1024) / g.aslot_bytes));
        g.h_tiles = (H + kTcTileM - 1) / kTcTileM;
        int32_t ctr = 0;
        const int32_t tq = (nq * d + kTcTileM - 1) / kTcTileM, tk = (nkv * d + kTcTileM - 1) / kTcTileM;
        const int32_t sub = g.tc_sub;
        g.tcg[OP_QKV] = make_tc_geom(H, (nq + 2 * nkv) * d, ctr, sub);
        g.tcg[OP_QKV].tiles = tq + 2 * tk;  // q, k and v tiled separately
        g.tcg[OP_QKV].units = g.tcg[OP_QKV].tiles * g.tcg[OP_QKV].kchunks;
        g.tcg[OP_QKV].tiles_q = tq;
        g.tcg[OP_QKV].tiles_k = tk;
        ctr += g.tcg[OP_QKV].tiles;
        g.tcg[OP_O] = make_tc_geom(nq * d, H, ctr, sub);
        ctr += g.tcg[OP_O].tiles;
        g.tcg[OP_GU] = make_tc_geom(H, I, ctr, sub);
        ctr += g.tcg[OP_GU].tiles;
        g.tcg[OP_DOWN] = make_tc_geom(I, H, ctr, sub);
        ctr += g.tcg[OP_DOWN].tiles;
        g.tcg[OP_LM] = make_tc_geom(H, V, ctr, sub);
        ctr += g.tcg[OP_LM].tiles;
        // ranges per projection: every CTA, or at most tc_tile_split per row tile
        for (int op : {OP_QKV, OP_O, OP_GU, OP_DOWN, OP_LM}) {
            TcGeom &t = g.tcg[op];
            t.nranges = opt.num_ctas;
            if (opt.tc_tile_split > 0)
                t.nranges = (int32_t)std::min<int64_t>(opt.num_ctas, (int64_t)t.tiles * opt.tc_tile_split);
        }
        g.n_tile_ctrs = ctr;
    }

    // CTA permutation (identity unless a planner seed is given)
    std::vector<int32_t> perm(N);
    std::iota(perm.begin(), perm.end(), 0);
    if (opt.planner_seed) {
        std::mt19937 rng(opt.planner_seed);
        std::shuffle(perm.begin(), perm.end(), rng);
    }

    // Work items of a projection: output rows (batch 1) or units (batched).
    auto items = [&](int32_t op) -> int32_t { return tc ? g.tcg[op].units : g.mv[op].rows; };

    std::vector<std::vector<Task>> q(N);
    // Dynamic dispatch (opt.jit): no task is bound to a CTA.  The tasks of
    // each stage (a layer's operator) sit together in stage order, and at run
    // time every CTA's scheduler claims the next unclaimed task of the
    // earliest unfinished stage.  Batch-1 projections are cut into jit ranges
    // per CTA, so that faster CTAs take more of them; the tensor-core path
    // keeps one range per CTA (its row-tile fixups are numbered by range).
    const bool jit = opt.jit > 0;
    const int32_t R = (jit && !tc) ? opt.jit * N : N;  // ranges per projection stage
    std::vector<Task> flat;
    std::vector<int32_t> stage_off;
    auto begin_stage = [&]() {
        if (jit) stage_off.push_back((int32_t)flat.size());
    };
    auto push = [&](const Task &t, int32_t c) {
        if (jit) flat.push_back(t);
        else q[perm[c % N]].push_back(t);
    };
    // Ranges of a stage: R, or the tensor-core projection's own count.
    auto ranges_of = [&](int32_t op) -> int32_t {
        return (tc && op != OP_EMBED && op != OP_KVA && g.tcg[op].nranges > 0) ? g.tcg[op].nranges : R;
    };
    // CTA after the last one the previous stage used: a stage that uses fewer
    // than every CTA starts there, so that small stages fall on the CTAs the
    // stage before left idle (or lightly loaded).
    int32_t cursor = 0;
    // Cuts `total` items into the stage's ranges (balanced to one item);
    // static dispatch gives range c to CTA perm[c] (perm[(cursor + c) % N]
    // for a stage of fewer than N ranges).  Returns the number of tasks.
    auto emit_ranges = [&](int32_t op, int32_t layer, int32_t total, uint16_t wait_ev, uint32_t wait_cnt,
                           uint16_t sig_ev) -> uint32_t {
        uint32_t n = 0;
        const int32_t Rop = ranges_of(op);
        const int32_t start = (Rop < N) ? cursor : 0;
        begin_stage();
        for (int32_t c = 0; c < Rop; ++c) {
            int32_t r0 = (int32_t)((int64_t)c * total / Rop), r1 = (int32_t)((int64_t)(c + 1) * total / Rop);
            if (r1 <= r0) continue;
            Task t{};
            t.op = (uint8_t)op;
            t.layer = (uint16_t)layer;
            t.wait_ev = wait_ev;
            t.wait_count = wait_cnt;
            t.signal_ev = sig_ev;
            t.a0 = r0;
            t.a1 = r1;
            t.a2 = c;
            push(t, start + c);
            ++n;
        }
        cursor = (int32_t)((start + n) % N);
        return n;
    };
    auto count_ranges = [&](int32_t op, int32_t total) { return (uint32_t)std::min<int64_t>(total, ranges_of(op)); };

    uint16_t x_ready_ev = kNoEvent;
    uint32_t x_ready_cnt = 0;
    if (tc) {
        // embedding rows and the first RMSNorm statistics, one item per (sequence, H tile)
        const uint16_t ev = (uint16_t)(per * L);
        x_ready_cnt = emit_ranges(OP_EMBED, 0, B * g.h_tiles, kNoEvent, 0, ev);
        x_ready_ev = ev;
    }
    const uint32_t n_qkv = count_ranges(OP_QKV, items(OP_QKV)), n_o = count_ranges(OP_O, items(OP_O)),
                   n_gu = count_ranges(OP_GU, items(OP_GU)), n_down = count_ranges(OP_DOWN, items(OP_DOWN));
    auto ev = [&](int32_t l, int32_t op) { return (uint16_t)ev_id(l, op, per); };
    for (int32_t l = 0; l < L; ++l) {
        uint32_t k = emit_ranges(OP_QKV, l, items(OP_QKV), x_ready_ev, x_ready_cnt, ev(l, OP_QKV));
        if (k != n_qkv) return MK_ERR_INVALID;
        // attention waits for every row's q (and, in kv-append graphs, for
        // every row's K/V in the cache: rows of one sequence attend to each other)
        uint16_t att_ev = ev(l, OP_QKV);
        uint32_t att_cnt = n_qkv;
        if (opt.kv_append) {
            att_cnt = emit_ranges(OP_KVA, l, B * nkv, ev(l, OP_QKV), n_qkv, ev(l, OP_KVA));
            att_ev = ev(l, OP_KVA);
        }
        // attention: one task per (sequence, kv head, split), round-robin over
        // CTAs in pair order (the pairs cut into more splits come last)
        begin_stage();
        int32_t i = 0;
        for (int32_t b = 0; b < B; ++b)
            for (int32_t h = 0; h < nkv; ++h) {
                const int32_t sp = psplit[b * nkv + h];
                for (int32_t s = 0; s < sp; ++s, ++i) {
                    Task t{};
                    t.op = OP_ATTN;
                    t.layer = (uint16_t)l;
                    t.wait_ev = att_ev;
                    t.wait_count = att_cnt;
                    t.signal_ev = ev(l, OP_ATTN);
                    t.a0 = b;
                    t.a1 = h;
                    t.a2 = s;
                    t.a3 = sp;
                    push(t, i);
                }
            }
        cursor = i % N;
        emit_ranges(OP_O, l, items(OP_O), ev(l, OP_ATTN), (uint32_t)(B * nkv), ev(l, OP_O));
        emit_ranges(OP_GU, l, items(OP_GU), ev(l, OP_O), n_o, ev(l, OP_GU));
        emit_ranges(OP_DOWN, l, items(OP_DOWN), ev(l, OP_GU), n_gu, ev(l, OP_DOWN));
        x_ready_ev = ev(l, OP_DOWN);
        x_ready_cnt = n_down;
    }
    emit_ranges(OP_LM, L - 1, items(OP_LM), x_ready_ev, x_ready_cnt, kNoEvent);

    if (opt.test_unreachable_event > 0) {
        const int32_t ev = opt.test_unreachable_event - 1;
        if (ev >= g.n_events) return MK_ERR_INVALID;
        for (auto &qq : q)
            for (Task &t : qq)
                if (t.wait_ev == ev) ++t.wait_count;
        for (Task &t : flat)
            if (t.wait_ev == ev) ++t.wait_count;
    }
    g.jit = jit;
    if (jit) {
        out->tasks = flat;
        stage_off.push_back((int32_t)flat.size());
        out->stage_off = stage_off;
        out->queue_off.assign(N + 1, 0);  // no task is bound to a CTA
        return MK_OK;
    }
    out->stage_off.clear();
    out->tasks.clear();
    out->queue_off.assign(N + 1, 0);
    for (int32_t c = 0; c < N; ++c) {
        out->queue_off[c] = (int32_t)out->tasks.size();
        out->tasks.insert(out->tasks.end(), q[c].begin(), q[c].end());
    }
    out->queue_off[N] = (int32_t)out->tasks.size();
    return MK_OK;
}

}  // namespace mk
