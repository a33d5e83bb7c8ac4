// mk_types.h — task-graph and kernel-parameter types shared by the host
// planner and the device runtime of the decode megakernel.
#pragma once

#include <stdint.h>

namespace mk {

enum Op : uint8_t { OP_NONE = 0, OP_QKV = 1, OP_ATTN = 2, OP_O = 3, OP_GU = 4, OP_DOWN = 5, OP_LM = 6, OP_COUNT = 7 };

constexpr uint16_t kNoEvent = 0xFFFF;

// One task of a worker CTA's queue.  A matvec task computes output rows
// [a0, a1) of its operator; an attention task covers one (sequence a0, kv
// head a1) pair over context split a2 of a3.
struct Task {
    uint8_t op;
    uint8_t flags;
    uint16_t layer;
    uint16_t wait_ev;     // kNoEvent: no dependency
    uint16_t signal_ev;   // kNoEvent: signals nothing
    uint32_t wait_count;  // proceed once counter[wait_ev] >= wait_count
    int32_t a0, a1, a2, a3;
    uint32_t pad[3];
};
static_assert(sizeof(Task) == 40, "task layout");

// Per-layer weight pointers (device copies of the caller's pointers).
struct LayerW {
    const uint16_t *attn_norm, *wq, *wk, *wv, *wo, *mlp_norm, *w_gate, *w_up, *w_down;
};

// How a matvec operator's weight rows are cut into ring slots: a slot holds
// `rpp` rows (times 2 for gate/up, which streams matching gate and up rows)
// of one column piece; a row is cut into `ksplit` pieces of at most `kc`
// columns when one row does not fit a slot.
struct MvGeom {
    int32_t K;        // input length (columns)
    int32_t rows;     // output rows of the operator
    int32_t rpp;      // rows per slot
    int32_t ksplit;   // column pieces per row
    int32_t kc;       // columns per piece (multiple of 8), last piece may be shorter
    int32_t row_mult; // 2 for gate/up, else 1
};

// Device error-word sites.
enum ErrSite : int32_t {
    SITE_NONE = 0,
    SITE_EVENT_WAIT = 1,
    SITE_READY_WAIT = 2,
    SITE_FULL_WAIT = 3,
    SITE_EMPTY_WAIT = 4,
    SITE_DRAIN_WAIT = 5,
    SITE_TOKEN = 6,
    SITE_POSITION = 7,
    SITE_PAGE = 8,
    SITE_ABORTED = 9,
};

// Layout of the plan's control words (uint32 each, zeroed at plan creation).
//   [0, n_events)                           event counters
//   [n_events, n_events + batch*n_kv_heads) attention split-done counters
//   then: exit counter, abort flag, error status, error site, error cta, error detail
struct CtlLayout {
    int32_t n_events;
    int32_t n_done;
    int32_t exit_idx, abort_idx, err_idx;
    int32_t total;
};

inline CtlLayout ctl_layout(int32_t n_events, int32_t n_done) {
    CtlLayout c;
    c.n_events = n_events;
    c.n_done = n_done;
    c.exit_idx = n_events + n_done;
    c.abort_idx = c.exit_idx + 1;
    c.err_idx = c.abort_idx + 1;
    c.total = c.err_idx + 4;
    return c;
}

}  // namespace mk
