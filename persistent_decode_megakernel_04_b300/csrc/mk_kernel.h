// mk_kernel.h — parameters and launchers of the decode megakernel.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_types.h"

namespace mk {

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kWarpSched = 0;
constexpr int kWarpProd = 1;
constexpr int kThreads = (2 + kComputeWarps) * 32;  // 320
constexpr int kMaxSlots = 16;
constexpr int kMaxGroup = 8;      // q heads per kv head
constexpr int kMaxHeadDim = 128;
constexpr int kMaxTps = 128;      // KV tokens per ring slot

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
    MvGeom mv[OP_COUNT];
    int32_t slot_bytes, num_slots, tps, attn_splits;
    int32_t l2_prefetch_bytes;
    // launch mode
    int32_t only_op;     // -1: every task (persistent mode); else one operator of one layer
    int32_t only_layer;
    int32_t skip_lm;     // prefill positions before the last: no LM head
    uint64_t timeout_ns;
    // optional task trace: [num_ctas][trace_stride][8] globaltimer stamps
    uint64_t *trace;
    int32_t trace_stride;
};

// Shared memory the megakernel needs for a given ring.
size_t megakernel_smem_bytes(int32_t slot_bytes, int32_t num_slots);

// Picks the register-tile variant for the longest matvec input.
int megakernel_variant(int32_t max_k);

// Launches the megakernel: cooperative (persistent mode) or plain (ablation).
cudaError_t launch_megakernel(const KParams &p, int variant, int grid, size_t smem, bool cooperative,
                              cudaStream_t stream);
cudaError_t megakernel_max_active(int variant, size_t smem, int *blocks_per_sm);
cudaError_t megakernel_set_smem(int variant, size_t smem);

cudaError_t launch_rope_table(float2 *rope, int32_t max_seq, int32_t d, float theta, cudaStream_t stream);
cudaError_t launch_greedy_next(const float *logits, int32_t B, int32_t V, int32_t *tokens, int32_t *positions,
                               cudaStream_t stream);

}  // namespace mk
