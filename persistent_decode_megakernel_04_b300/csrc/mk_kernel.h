// mk_kernel.h — parameters and launchers of the decode megakernel.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mk.h"
#include "mk_types.h"

namespace mk {

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kWarpSched = 0;
constexpr int kWarpProd = 1;
constexpr int kThreads = (3 + kComputeWarps) * 32;  // 352: scheduler, producer, 8 compute warps, MMA warp
constexpr int kMaxSlots = 16;
constexpr int kMaxGroup = 8;      // q heads per kv head
constexpr int kMaxHeadDim = 128;
constexpr int kAttnBlock = 64;    // cached tokens per attention block (one aligned run of a page)
constexpr int kQhlStride = kMaxHeadDim + 8;  // bf16 row stride of the split queries (conflict-free ldmatrix)
constexpr int kAttnStep = 2 * kAttnBlock;    // cached tokens an attention step handles at most
constexpr int kPhlStride = kAttnStep + 8;    // bf16 row stride of the split softmax weights
constexpr int kMaxResid = 512;    // residual rows prefetched per matvec task
constexpr int kMvResident = 2;    // matvec inputs of up to 2 x 2048 columns stay in registers
constexpr int kMvSuper = 2;       // longer inputs: row groups that stream piece by piece together, so that
                                  // each input piece is loaded once for all of them
constexpr int kMaxASlots = 8;     // activation ring slots (batched path)
constexpr int kJitRing = 8;       // dynamic dispatch: ring slots of claimed tasks
constexpr int kJitAhead = 1;      // dynamic dispatch: claims beyond the task the compute warps hold

struct KParams {
    // shape
    int32_t L, H, nq, nkv, d, I, V, B, max_seq, page_size;
    float eps;
    int32_t qkv_rows;
    // weights
    const uint16_t *embed, *lm_head, *final_norm;
    const LayerW *layers;
    // KV cache
    uint16_t *k_pool, *v_pool;
    const int32_t *page_table;
    int32_t num_pages, max_pages;
    int32_t pt_stride;     // page-table entries between batch rows (0: every row is one sequence)
    int32_t kv_appended;   // OP_KVA tasks append the new K/V; attention reads positions 0..pos from the cache
    // inputs / outputs of this step
    const int32_t *tokens;
    int32_t tok_stride;
    const int32_t *positions;
    int32_t pos_stride;
    float *logits;
    // plan scratch
    float *x, *qkv, *attn_part, *attn_out, *hbuf;
    const float2 *rope;  // [max_seq][d/2] (cos, sin)
    uint32_t *ctl;       // control words, see CtlLayout
    CtlLayout cl;
    // task graph
    const Task *tasks;
    const int32_t *queue_off;
    // dynamic dispatch (0: static queues): stage s holds tasks
    // [stage_off[s], stage_off[s + 1]); claim counters at ctl + cl.claim_idx
    int32_t jit;
    int32_t n_stages;
    const int32_t *stage_off;
    MvGeom mv[OP_COUNT];
    int32_t slot_bytes, num_slots, attn_ts, attn_splits;  // attn_ts: KV tokens per ring slot
    int32_t l2_prefetch_bytes;
    int32_t max_inflight;  // ring copies in flight per CTA (0 or >= num_slots: no limit)
    // batch 1: per-layer tensor maps of w_down seen as [H][I/256][256] bf16,
    // boxes of rpp rows x kc/256 blocks x 256 columns, so that one TMA copy
    // fills a ring slot with piece ks of a row group (nullptr: one bulk copy
    // per row and piece)
    const uint8_t *down_maps;
    // launch mode
    int32_t only_op;     // -1: every task (persistent mode); else one operator of one layer
    int32_t only_layer;
    int32_t skip_lm;     // prefill positions before the last: no LM head
    // batch 1, fused greedy pick: after the LM head, next_tokens[0] = argmax
    // of the logits (lowest index among equal maxima), next_positions[0] += 1
    int32_t greedy;
    int32_t *next_tokens, *next_positions;
    uint64_t timeout_ns;
    // optional task trace: [num_ctas][trace_stride][8] globaltimer stamps
    uint64_t *trace;
    int32_t trace_stride;
    // TMA maps of the K and V pools seen as [L*num_pages*nkv*page_size][d]
    // bf16 rows, boxes of 64 columns x attn_ts rows, 128-byte swizzled
    alignas(64) uint8_t kv_maps[2][128];
    int32_t kv_halves_3d;  // kv_maps are 3-D views copying both 64-column halves of d = 128 at once
    // batched (tensor-core) path
    int32_t tc;              // nonzero: projections run as tcgen05 tiles
    int32_t npad;            // MMA N: batch rounded up to 16
    uint32_t idesc;          // kind::f16 instruction descriptor (M 128, N npad)
    int32_t num_ctas;        // ranges per projection
    int32_t h_tiles;         // 128-row tiles of the hidden size
    int32_t aslot_bytes, num_aslots;
    int32_t tc_sub;  // 64-column K sub-tiles per projection unit (one ring slot, one activation slot)
    uint32_t tmem_cols;
    TcGeom tcg[OP_COUNT];
    const uint8_t *tmaps;    // CUtensorMap[7 * L + 4], see the kernel's TmIdx
    uint16_t *xa;            // bf16 [B][H]: x times the next consumer's RMSNorm gain
    float *ssq;              // fp32 [B][h_tiles]: sums of x^2 over 128-row tiles of x
    uint16_t *attn_a;        // bf16 [B][nq*d]: attention output
    uint16_t *h_a;           // bf16 [B][I]: SiLU(gate) * up
    float *part;             // fp32 [num_ctas][2][2][npad][128]: partial row-tile sums
    uint32_t *tile_ctr;      // row-tile arrival counters
};

// Shared memory the megakernel needs for a given ring (plus the activation
// ring of the batched path).
size_t megakernel_smem_bytes(int32_t slot_bytes, int32_t num_slots, int32_t aslot_bytes, int32_t num_aslots);

// Picks the kernel build: static queues or dynamic dispatch.
int megakernel_variant(int32_t max_k, bool tc, bool jit);

// Launches the megakernel: cooperative (persistent mode) or plain (ablation).
cudaError_t launch_megakernel(const KParams &p, int variant, int grid, size_t smem, bool cooperative,
                              cudaStream_t stream);
cudaError_t megakernel_max_active(int variant, size_t smem, int *blocks_per_sm);
// Raises the kernel's dynamic shared-memory limit to at least smem (never
// lowers it: the limit is shared by every plan and call in the process).
cudaError_t megakernel_set_smem(int variant, size_t smem);

// Host: TMA maps of the K and V pools (KParams::kv_maps) for tiles of ts tokens.
bool encode_kv_maps(KParams &k, const mk_model_cfg &c, const mk_kv_cache &kv, int32_t ts);

// Host: whether batch-1 down-projection slots can come from one 3-D TMA copy
// each (pieces of 2048 columns, rows a multiple of them), and the map of one
// layer's w_down (128 bytes at m).
bool down_tma_ok(const MvGeom &g);
bool encode_down_map(void *m, const void *w_down, const MvGeom &g);

cudaError_t launch_rope_table(float2 *rope, int32_t max_seq, int32_t d, float theta, cudaStream_t stream);
cudaError_t launch_greedy_next(const float *logits, int32_t B, int32_t V, int32_t *tokens, int32_t *positions,
                               cudaStream_t stream);

// Rows of one chunked-prefill launch: tok[j] = src[min(j, n-1)] and
// pos[j] = p0 + min(j, n-1) for j < rows.
cudaError_t launch_prefill_rows(const int32_t *src, int32_t n, int32_t p0, int32_t rows, int32_t *tok, int32_t *pos,
                                cudaStream_t stream);

}  // namespace mk
