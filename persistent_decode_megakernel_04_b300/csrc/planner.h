// planner.h — host task-graph builder of the decode megakernel.
#pragma once

#include <vector>

#include "../../include/mk.h"
#include "mk_types.h"

namespace mk {

struct PlanGeom {
    int32_t num_ctas = 0;
    int32_t attn_splits = 0;
    int32_t slot_bytes = 0;
    int32_t num_slots = 0;
    int32_t tps = 0;  // KV tokens per ring slot (divides the 64-token attention block)
    int32_t n_events = 0;
    int32_t l2_prefetch_bytes = 0;
    int32_t max_inflight = 0;  // ring copies in flight per CTA (0: no limit)
    bool kv_append = false;    // K/V appended by OP_KVA tasks before attention
    bool jit = false;          // dynamic dispatch: CTAs claim tasks stage by stage at run time
    MvGeom mv[OP_COUNT] = {};
    // batched (tensor-core) path
    bool tc = false;
    int32_t npad = 0;         // batch rounded up to the MMA N granule (16)
    int32_t tc_sub = 1;       // 64-column K sub-tiles per projection unit (ring slot)
    int32_t aslot_bytes = 0;  // activation ring slot: npad rows x 64 bf16
    int32_t num_aslots = 0;
    int32_t h_tiles = 0;      // 128-row tiles of the hidden size
    int32_t n_tile_ctrs = 0;  // row-tile counters of all projections
    TcGeom tcg[OP_COUNT] = {};
};

struct PlanTables {
    PlanGeom g;
    std::vector<Task> tasks;          // CTA 0's queue, then CTA 1's, ... (dynamic dispatch: stage by stage)
    std::vector<int32_t> queue_off;   // [num_ctas + 1]
    std::vector<int32_t> stage_off;   // dynamic dispatch: first task of each stage, then the task count
};

// Fills in defaults for zero option fields.
mk_plan_options resolve_options(const mk_model_cfg &cfg, const mk_plan_options *opt, int32_t num_sms);

// Shape checks shared by plan creation and the host-only describe call.
mk_status check_cfg(const mk_model_cfg &cfg);

// Builds the task graph for cfg on opt.num_ctas worker CTAs.
mk_status build_plan(const mk_model_cfg &cfg, const mk_plan_options &opt, PlanTables *out);

// Event ids: per layer QKV, ATTN, O, GU, DOWN, then KV-APPEND in graphs
// that append K/V in a task of their own (per = 6; otherwise per = 5).
inline int32_t ev_id(int32_t layer, int32_t op, int32_t per) {
    return layer * per + (op == OP_KVA ? 5 : op - 1);
}

}  // namespace mk
