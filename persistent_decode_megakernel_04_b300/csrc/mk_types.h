// mk_types.h — task-graph and kernel-parameter types shared by the host
// planner and the device runtime of the decode megakernel.
#pragma once

#include <stdint.h>

namespace mk {

enum Op : uint8_t {
    OP_NONE = 0, OP_QKV = 1, OP_ATTN = 2, OP_O = 3, OP_GU = 4, OP_DOWN = 5, OP_LM = 6,
    OP_EMBED = 7,  // batched path only: embedding rows + first RMSNorm statistics
    OP_KVA = 8,    // kv-append graphs only: RoPE + bf16 append of every row's new K/V before attention
    OP_COUNT = 9
};

constexpr uint16_t kNoEvent = 0xFFFF;
constexpr int32_t kMaxSplits = 64;  // attention context splits per (sequence, kv head)

// One task of a worker CTA's queue.  A matvec task computes output rows
// [a0, a1) of its operator; an attention task covers one (sequence a0, kv
// head a1) pair over context split a2 of a3.  On the batched path a
// projection task covers units [a0, a1) of its operator (see TcGeom) as
// range number a2, and an embedding task covers items [a0, a1) (item =
// sequence * H-tiles + H-tile).
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

// How a matvec operator's weight rows are cut into ring slots.  A row is
// cut into `ksplit` pieces of `kc` columns (the last may be shorter); each
// compute thread owns column chunk ct of every piece.  Rows are processed in
// groups of `rpp` (gate/up: rpp gate rows and the matching up rows).
//  - Whole-row slots (rps > 0, inputs of at most 4096 columns): a slot holds
//    rps consecutive whole rows of one matrix, one contiguous copy.
//  - Piece slots (rps == 0): a slot holds piece ks of the group's rows
//    (gate rows, then up rows).
struct MvGeom {
    int32_t K;        // input length (columns)
    int32_t rows;     // output rows of the operator
    int32_t rpp;      // rows per group (of each matrix, for gate/up)
    int32_t ksplit;   // column pieces per row
    int32_t kc;       // columns per piece (2048, or K when K is shorter)
    int32_t row_mult; // 2 for gate/up, else 1
    int32_t rps;      // whole-row slots: rows of one matrix per slot (4 or 8); 0: piece slots
};

// Batched path: an operator's weight [rows x K] is cut into units of
// kTcTileM rows x kTcTileK columns (one tcgen05 A tile); unit u is row tile
// u / kchunks, column chunk u % kchunks.  Each worker CTA owns one
// contiguous range of units (the ranges are balanced to one unit), so a row
// tile can be shared by several CTAs, whose fp32 partial sums the last one
// to finish adds up in range order.  The q, k and v matrices are tiled
// separately: row tiles [0, tiles_q) are q, [tiles_q, tiles_q + tiles_k) k,
// the rest v.
constexpr int32_t kTcTileM = 128;
constexpr int32_t kTcTileK = 64;
constexpr int32_t kTcMaxBatch = 64;  // MMA N = 2 * npad <= 128; TMEM holds 2 buffers x 2 matrices

struct TcGeom {
    int32_t K, rows;
    int32_t tiles, kchunks, units;
    int32_t tiles_q, tiles_k;  // QKV only
    int32_t ctr_off;           // first row-tile counter of this operator
    int32_t nranges;           // contiguous balanced ranges the units are cut into (one per task)
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
    SITE_ACC_WAIT = 10,
};

// Layout of the plan's control words (uint32 each, zeroed at plan creation).
//   [0, n_events)                           event counters
//   [n_events, n_events + batch*n_kv_heads) attention split-done counters
//   then n_claims claim counters (dynamic dispatch), n_tiles row-tile
//   counters (batched path), then: exit counter, abort
//   flag, error status, error site, error cta, error detail, then one 64-bit
//   word per sequence (even index): the fused greedy pick's packed maximum
struct CtlLayout {
    int32_t n_events;
    int32_t n_done;
    int32_t claim_idx, n_claims;  // dynamic dispatch: one claim counter per stage
    int32_t tile_idx, n_tiles;
    int32_t exit_idx, abort_idx, err_idx;
    int32_t amax_idx;  // sequence b's packed (logit, index) maximum: words amax_idx + 2b, + 2b + 1
    int32_t total;
};

inline CtlLayout ctl_layout(int32_t n_events, int32_t n_done, int32_t n_tiles, int32_t n_seq, int32_t n_claims = 0) {
    CtlLayout c;
    c.n_events = n_events;
    c.n_done = n_done;
    c.claim_idx = n_events + n_done;
    c.n_claims = n_claims;
    c.tile_idx = c.claim_idx + n_claims;
    c.n_tiles = n_tiles;
    c.exit_idx = c.tile_idx + n_tiles;
    c.abort_idx = c.exit_idx + 1;
    c.err_idx = c.abort_idx + 1;
    c.amax_idx = (c.err_idx + 4 + 1) & ~1;
    c.total = c.amax_idx + 2 * n_seq;
    return c;
}

}  // namespace mk
