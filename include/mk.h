/*
 * mk.h — C ABI of the persistent decode megakernel for B300 (sm_103a).
 *
 * One decode step of a Llama-style decoder (RMSNorm, QKV projection, RoPE,
 * GQA attention over a paged bf16 KV cache, O-projection + residual, SwiGLU
 * MLP, LM head) runs as ONE cooperative kernel launch.  Inside it, every SM
 * hosts one worker CTA with a scheduler warp, a weight-streaming producer
 * warp and eight compute warps; tasks are ordered by global-memory event
 * counters, never by kernel boundaries or grid-wide barriers.
 *
 * Where each operation is defined (page titles and sections):
 *  - single-kernel execution of the whole step, task graph of per-SM tasks
 *    and events, worker loop, scheduler warps, counter-with-threshold events:
 *    "Compilar LLM en un MegaKernel para lograr inferencia de baja latencia"
 *    (es.news.hada.io/topic?id=21563), sections "Parte 1. Compilador",
 *    "Parte 2. Runtime", "Método de ejecución basado en eventos";
 *  - the tGraph of SM-level tasks, ahead-of-time task preparation and the
 *    paged shared memory that lets the next task's data load while the
 *    current one finishes: "MPK: A Compiler and Runtime for Mega-Kernelizing
 *    Tensor Programs" (gist.science/fr/paper/2512.22219), sections 2–4;
 *  - the fused instructions (RMS norm, QKV matmul + RoPE, attention, O-proj
 *    matmul + residual), matrix-vector tasks for low latency and
 *    matrix-matrix tasks for throughput: "Llama-70B 向け…megakernel"
 *    (hakusoku.com/story/2591), section 高スループットMegakernelの設計と工夫;
 *  - residual + norm fusion and the fused SwiGLU feed-forward: "Cómo la
 *    fusión de kernels CUDA acelera la inferencia de LLM" (slavadubrov.com),
 *    section "Sigue los datos intermedios".
 *
 * Conventions for every function below:
 *  - Memory: weights, KV pools, page table, tokens, positions and logits are
 *    CALLER-OWNED device memory (unless a name ends in _host) and must stay
 *    valid until the work queued on `stream` has finished.  The plan owns its
 *    scratch, event counters, task tables, RoPE table and error word.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on it unless stated otherwise.
 *  - Errors that the host can detect return synchronously and launch nothing.
 *    Errors found on the device (a wait that exceeded the plan's time budget,
 *    an out-of-range token, position or page id) are recorded in the plan's
 *    device error word; the kernel then exits without faulting.  Read them
 *    with mk_plan_last_error.  The error stays set (and later steps return
 *    early on the device) until mk_plan_last_error clears it.
 *  - One plan is used by one stream at a time; calls that overlap on the GPU
 *    race on the plan's scratch.
 */
#ifndef MK_H
#define MK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MK_OK = 0,
    MK_ERR_INVALID = 1,     /* bad argument, null or misaligned pointer, bad shape */
    MK_ERR_CUDA = 2,        /* a CUDA runtime call failed */
    MK_ERR_LAUNCH = 3,      /* the cooperative grid cannot be co-resident */
    MK_ERR_TIMEOUT = 4,     /* a device wait exceeded the plan's time budget */
    MK_ERR_BOUNDS = 5,      /* token, position or page id out of range (device) */
    MK_ERR_OOM = 6,         /* plan scratch allocation failed */
    MK_ERR_UNSUPPORTED = 7  /* shape outside what this build implements */
} mk_status;

/* Decoder shape and the plan's fixed batch/context geometry. */
typedef struct {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    float rms_eps, rope_theta;
    int32_t tied_embeddings; /* nonzero: lm_head == embed */
    int32_t batch;           /* sequences per step, fixed per plan (1: CUDA-core matvec path;
                                2..64: tensor-core path) */
    int32_t max_seq;         /* positions 0..max_seq-1 are valid */
    int32_t page_size;       /* tokens per KV page */
} mk_model_cfg;

/* Weights: bf16, row-major [out][in], 16-byte aligned device pointers.
 * Per-layer entries are HOST arrays of n_layers device pointers.
 * Shapes: embed/lm_head [vocab][hidden]; final_norm, attn_norm, mlp_norm
 * [hidden]; wq [n_q_heads*head_dim][hidden]; wk, wv [n_kv_heads*head_dim]
 * [hidden]; wo [hidden][n_q_heads*head_dim]; w_gate, w_up [ffn_dim][hidden];
 * w_down [hidden][ffn_dim].  Not modified and not copied: the plan keeps the
 * pointers, so the weights must outlive the plan. */
typedef struct {
    const void *embed, *lm_head, *final_norm;
    const void *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo;
    const void *const *mlp_norm, *const *w_gate, *const *w_up, *const *w_down;
} mk_weight_ptrs;

/* Paged KV cache (caller-owned).  Pools are bf16
 * [n_layers][num_pages][n_kv_heads][page_size][head_dim]; page_table is a
 * device int32 [batch][max_pages_per_seq]: token t of sequence b lives in
 * page page_table[b][t / page_size], slot t % page_size. */
typedef struct {
    void *k_pool, *v_pool;
    const int32_t *page_table;
    int32_t num_pages, max_pages_per_seq;
} mk_kv_cache;

/* Optional plan knobs; zero fields take the defaults. */
typedef struct {
    int32_t num_ctas;      /* worker CTAs (default: every SM) */
    int32_t attn_splits;   /* context splits per (sequence, kv head), at most 64
                              (default: CTAs / (batch*n_kv_heads), capped at 64).  With one
                              split and more pairs than CTAs, the pairs left over after whole
                              rounds of CTAs are cut into the split count that evens the
                              CTAs' shares (static dispatch) */
    int32_t slot_bytes;    /* shared-memory ring slot size (default 32768) */
    int32_t num_slots;     /* ring slots (default 6 at batch 1; batched: as many as shared memory holds) */
    int32_t timeout_ms;    /* budget of every device wait (default 2000) */
    uint32_t planner_seed; /* nonzero: permute the CTA <-> tile assignment */
    int32_t l2_prefetch_kb;/* batch 1: on reaching an O projection, prefetch into L2 up to this many
                              KB of the weights the ring cannot hold yet (the O rows past the ring,
                              then the first gate/up rows); default 0 = off (measured slower) */
    int32_t test_unreachable_event; /* failure-path testing: k > 0 makes the waiters of event k-1
                                       need one signal more than can ever arrive, so their
                                       bounded wait expires and the step reports MK_ERR_TIMEOUT */
    int32_t trace;         /* nonzero: record per-task timestamps (see mk_plan_trace) */
    int32_t tensor_cores;  /* 0: projections as CUDA-core matvecs at batch 1, tcgen05 tiles at
                              batch >= 2; 1: tcgen05 tiles at every batch */
    int32_t max_inflight;  /* ring copies a CTA keeps in flight at once (default: 3 at batch 1,
                              every free ring slot when batched; >= num_slots: no cap) */
    int32_t kv_append;     /* 1: a task of its own (op 8) RoPEs and appends every row's new K/V
                              to the cache before attention, which then reads the new token from
                              the cache like the rest; rows may then be consecutive tokens of one
                              sequence (the chunked-prefill graph of mk_prefill).  Default 0: the
                              last attention split appends its row's K/V itself */
    int32_t prefill_by_decode; /* 1: mk_prefill runs the decode step once per position instead of
                                  the chunked-prefill engine */
    int32_t jit;           /* 0: static dispatch, every task bound to a CTA ahead of time (default);
                              n >= 1: dynamic dispatch: each CTA's scheduler warp claims the next
                              unclaimed task of the earliest unfinished stage (a layer's operator)
                              at run time, batch-1 projections cut into n ranges per CTA (at most
                              16; the tensor-core path keeps one range per CTA).  Not with trace;
                              the ablation build needs static dispatch */
    int32_t test_poison_scratch; /* testing: nonzero fills every activation buffer of the plan's
                                    scratch with 0xFF bytes (NaN as fp32 and as bf16) before each
                                    step, so that a value a step reads without having written it
                                    shows up as NaN in the logits; costs a memset per buffer */
    int32_t tc_tile_split; /* tensor-core path: at most this many worker CTAs share one 128-row
                              tile of a projection; small projections then run on fewer CTAs
                              with fewer partial sums to add (0: every CTA takes a range of
                              every projection) */
    int32_t tc_k_subtiles; /* tensor-core path: 64-column K sub-tiles per projection unit (ring
                              slot), 1 or 2; two halve the waits and commits per weight byte
                              but make slots twice as large (0: 2) */
    int32_t reserved[1];
} mk_plan_options;

typedef struct mk_plan mk_plan; /* opaque, library-owned */

/* Device error report. */
typedef struct {
    int32_t status; /* mk_status of the first device error, MK_OK if none */
    int32_t site;   /* where it happened (see mk_error_site_string) */
    int32_t cta;    /* worker CTA that recorded it */
    int32_t detail; /* event id, task index or offending value */
} mk_device_error;

/* Build a plan for one decoder and batch geometry on the current device.
 * Passage: the ahead-of-time task graph of "MPK: A Compiler and Runtime for
 * Mega-Kernelizing Tensor Programs", sections 2-3 (tGraph, AOT preparation),
 * and "Compilar LLM en un MegaKernel…", "Parte 1. Compilador".
 * Validates the shape and pointer alignment, builds the task graph (per-CTA
 * task queues and event thresholds), allocates the plan's scratch and
 * checks that the cooperative grid fits.  Synchronous.  *out is set only on
 * MK_OK.  MK_ERR_UNSUPPORTED: a shape this build does not implement. */
mk_status mk_plan_create(const mk_model_cfg *cfg, const mk_weight_ptrs *w, mk_plan **out);
mk_status mk_plan_create_ex(const mk_model_cfg *cfg, const mk_weight_ptrs *w, const mk_plan_options *opt,
                            mk_plan **out);

/* One decode step for every sequence of the batch.  Passage: the single
 * persistent launch of "Compilar LLM en un MegaKernel…", sections "Parte 2.
 * Runtime" and "Método de ejecución basado en eventos"; the fused task list
 * of "Llama-70B 向け…megakernel", section 高スループットMegakernelの設計と工夫.
 * tokens[b] at position
 * positions[b] (device int32 [batch]).  Appends K/V of that position to the
 * cache, attends over positions 0..positions[b], writes logits (device fp32
 * [batch][vocab]).  One cooperative launch. */
mk_status mk_decode_step(mk_plan *plan, const int32_t *tokens, const int32_t *positions, const mk_kv_cache *kv,
                         float *logits, void *stream);

/* Passage: the separate-kernel baseline that "Compilar LLM en un
 * MegaKernel…" compares against ("Limitaciones previas"), and the
 * measurement checklist of "Cómo la fusión de kernels CUDA acelera…",
 * "Comprueba si la fusión ha ayudado".
 * The same step, with the same task code, launched one kernel per operator
 * and layer (5 per layer + 1), ordered by the stream instead of by event
 * counters.  The launch-per-operator ablation of the megakernel. */
mk_status mk_decode_step_ablation(mk_plan *plan, const int32_t *tokens, const int32_t *positions,
                                  const mk_kv_cache *kv, float *logits, void *stream);

/* Passage: as mk_decode_step (a serving loop's view of one step).
 * mk_decode_step with HOST buffers: copies tokens/positions (host int32
 * [batch]) in, runs the step, copies logits (host fp32 [batch][vocab]) out
 * and synchronises `stream`.  Returns device errors of this step directly. */
mk_status mk_decode_step_host(mk_plan *plan, const int32_t *tokens_host, const int32_t *positions_host,
                              const mk_kv_cache *kv, float *logits_host, void *stream);

/* Passage: the prompt phase before decoding ("Compilar LLM en un
 * MegaKernel…", "Valor central de MPK": a 39-token prompt, then 512 decode
 * steps), and the comparison of small-batch decode with large-batch prefill
 * of "Cómo la fusión de kernels CUDA acelera…", "Comprueba si la fusión ha
 * ayudado".
 * Prefill T prompt tokens per sequence (device int32 [batch][T]) at
 * positions 0..T-1; writes the logits of position T-1 (device fp32
 * [batch][vocab]); the LM head runs only for the last chunk or position.
 * Plans of fewer than 64 sequences use a chunked-prefill engine: up to 64
 * consecutive tokens of one sequence per persistent launch, as the rows of
 * the tensor-core path, with a task that appends every row's K/V to the cache
 * before the rows attend (causally) to it.  The engine is a second plan of
 * the same weights, made (allocating device memory) on the first call;
 * options.prefill_by_decode, or a failure to make it, selects the decode
 * step once per position instead, as batched plans always do. */
mk_status mk_prefill(mk_plan *plan, const int32_t *tokens, int32_t T, const mk_kv_cache *kv, float *last_logits,
                     void *stream);

/* Passage: the throughput regime of "Llama-70B 向け…megakernel", section
 * 高スループットMegakernelの設計と工夫 (large batches of sequences that arrive
 * and leave), on one GPU.
 * Prefill the T prompt tokens (device int32 [T]) of ONE batch row at
 * positions 0..T-1, into the pages its page-table row names, with the
 * chunked-prefill engine (made on first use, allocating device memory),
 * whatever the plan's batch; the other rows' cache entries are untouched.
 * Writes the logits of position T-1 (device fp32 [vocab]).  Continuous
 * batching admits a sequence into a free row with this call. */
mk_status mk_prefill_row(mk_plan *plan, int32_t row, const int32_t *tokens, int32_t T, const mk_kv_cache *kv,
                         float *logits, void *stream);

/* Passage: greedy decoding of the measured runs ("Valor central de MPK").
 * Greedy continuation for the next step: tokens[b] = argmax_v logits[b][v]
 * (lowest index on ties) and positions[b] += 1, on the device. */
mk_status mk_greedy_next(mk_plan *plan, const float *logits, int32_t *tokens, int32_t *positions, void *stream);

/* Passage: the fused LM-head epilogue of "Cómo la fusión de kernels CUDA
 * acelera…", section "Sigue los datos intermedios".
 * One decode step followed by the greedy pick, in place: tokens[b] becomes
 * the argmax of row b of logits (the lowest index among equal maxima; NaN
 * never wins, and a row without a finite maximum gives 0x7FFFFFFF) and
 * positions[b] is incremented, exactly as mk_decode_step then
 * mk_greedy_next.  The pick runs inside the decode launch: at batch 1 (each
 * CTA's maximum over its LM-head rows, merged with one 64-bit atomic max);
 * batched plans pick in the tensor-core LM-head epilogue (each tile's best
 * row per sequence, one 64-bit atomic max per sequence and CTA), and the last
 * CTA out writes the tokens.  tokens and positions are
 * device arrays [batch], read by the step and rewritten after it; logits are
 * still written.  Errors as mk_decode_step. */
mk_status mk_decode_step_greedy(mk_plan *plan, int32_t *tokens, int32_t *positions, const mk_kv_cache *kv,
                                float *logits, void *stream);

/* Passage: token-by-token greedy generation ("Compilar LLM en un
 * MegaKernel…", "Valor central de MPK"), driven from host memory.
 * mk_decode_step_greedy with HOST buffers: copies tokens and positions (host
 * int32 [batch]) in, runs the step with the pick inside the launch, copies
 * the picked tokens (host int32 [batch]) out and synchronises `stream`.  The
 * logits stay in plan-owned device memory; positions_host is not changed
 * (the next step passes positions + 1).  Returns device errors of this step
 * directly. */
mk_status mk_decode_step_greedy_host(mk_plan *plan, const int32_t *tokens_host, const int32_t *positions_host,
                                     const mk_kv_cache *kv, int32_t *next_tokens_host, void *stream);

/* Passage: the 1-2 us task-switch cost that "Compilar LLM en un
 * MegaKernel…" reports ("Método de ejecución basado en eventos"); this call
 * measures it.
 * Task trace of the last step run with a plan created with options.trace:
 * for every CTA c and queue position i (the order of mk_plan_describe),
 * out[(c * *max_tasks + i) * 8 + k] holds, in globaltimer nanoseconds,
 *   k=0 scheduler released the task (its event reached the threshold),
 *   k=1 compute warps started it, k=2 they finished it,
 *   k=3 total time the compute warps waited for ring slots to fill,
 *   k=4 producer issued the task's first copy,
 *   k=5 total time the producer waited for free ring slots,
 *   k=6 (batched projections) total time the MMA issuer waited for
 *       activation tiles, k=7 ... for a free TMEM accumulator.
 * On the batched path k=3 of a projection task is the MMA issuer's wait for
 * weight tiles (the MMA warp's).  For attention tasks k=6 is the time spent
 * in slot waits and scores, k=7 the time in value sums (the rest is softmax
 * and per-task work); on the warp-local path of long splits k=6 is the whole
 * loop and k=3 the first compute warp's waits for its own slots.
 * Zeros mark tasks not run.  Synchronises `stream`.  Host buffer of
 * `capacity` uint64 values; MK_ERR_INVALID if tracing is off or the buffer is
 * too small (*max_tasks is still set). */
mk_status mk_plan_trace(mk_plan *plan, void *stream, uint64_t *out, int64_t capacity, int32_t *num_ctas,
                        int32_t *max_tasks);

/* Batch-1 decode step that allocates no device memory.
 *
 * The pages have no counterpart to this call. It exists for callers that
 * cannot call cudaMalloc when they need a decode step: code running while a
 * caching allocator or memory pool holds all of the device's free memory, a
 * runtime that reserves all device memory up front, or a serving process
 * that must not grow its footprint once it is serving. It needs no plan.
 * Each call builds the task graph on the host from `cfg` (batch must be 1;
 * other values return MK_ERR_UNSUPPORTED), then runs the same persistent
 * kernel as mk_decode_step, with the same arguments and results.
 *
 * Scratch: every call uses one fixed 16 MiB device array, compiled into this
 * library. Every GPU that loads the library holds those 16 MiB until the
 * process exits. A shape whose task tables, activations, attention partials
 * and RoPE table (max_seq x head_dim/2 x 8 bytes) need more returns MK_ERR_OOM
 * before anything is launched. The array keeps the last call's contents, so
 * each call uploads its tables and clears its counters and error word before
 * the launch. Calls that overlap on the GPU (on two streams at once) share the
 * array and race: issue them one at a time.
 *
 * The first call on a device (and the first after the device's context has
 * been replaced, for example by cudaDeviceReset) looks up the array's device
 * address on that device with cudaGetSymbolAddress. Make that first call
 * before any stream capture. The call calls no cudaMalloc or cudaFree.
 *
 * The call is synchronous: it waits for `stream` before it returns, and
 * returns the step's device-detected error (MK_ERR_BOUNDS, MK_ERR_TIMEOUT), if
 * any, as its status. weights, tokens, positions, kv and logits are as for
 * mk_plan_create and mk_decode_step. */
mk_status mk_decode_step_noalloc(const mk_model_cfg *cfg, const mk_weight_ptrs *w, const int32_t *tokens,
                                 const int32_t *positions, const mk_kv_cache *kv, float *logits, void *stream);

/* ---------------------------------------------------------------------
 * Continuous batching: a host-side allocator of the KV pool's pages and of
 * the batch's page table (no GPU needed except for mk_pages_sync).
 * Passage: the serving regime of "Llama-70B 向け…megakernel", section
 * 高スループットMegakernelの設計と工夫 (sequences of different lengths
 * sharing large decode batches), on one GPU.
 *
 * A plan's batch is a fixed set of rows.  Between decode steps a sequence is
 * admitted into a free row (pages for its prompt), grows page by page as it
 * decodes (mk_pages_extend before the step that writes a position its
 * pages do not cover) and retires, its pages going back to the pool.  The
 * pool's last page is scratch: every entry of a free row names it, so a
 * decode step over the whole batch may run a free row (token 0, position 0)
 * without touching any sequence's pages.  Errors: MK_ERR_INVALID for a bad
 * row or state (admitting a live row, extending or retiring a free one, a
 * length past max_pages_per_seq pages), MK_ERR_OOM when the pool has too
 * few free pages (nothing is allocated then).
 * --------------------------------------------------------------------- */
typedef struct mk_page_pool mk_page_pool; /* opaque, host-side */

/* num_pages: pages of the KV pools (the last one becomes scratch). */
mk_status mk_pages_create(int32_t num_pages, int32_t batch, int32_t max_pages_per_seq, int32_t page_size,
                          mk_page_pool **out);
/* Row becomes live with pages for its first n_tokens positions. */
mk_status mk_pages_admit(mk_page_pool *pool, int32_t row, int32_t n_tokens);
/* A live row's pages cover its first n_tokens positions (no-op if they do). */
mk_status mk_pages_extend(mk_page_pool *pool, int32_t row, int32_t n_tokens);
/* A live row's pages return to the pool; its entries name the scratch page. */
mk_status mk_pages_retire(mk_page_pool *pool, int32_t row);
int32_t mk_pages_free_count(const mk_page_pool *pool);
int32_t mk_pages_scratch_page(const mk_page_pool *pool);
/* Host copy of the page table, int32 [batch][max_pages_per_seq]. */
mk_status mk_pages_table(const mk_page_pool *pool, int32_t *out, int64_t capacity);
/* Copies the page table (if it changed since the last sync) to the device
 * table (int32 [batch][max_pages_per_seq]) on `stream`; the host copy may
 * change again as soon as the call returns. */
mk_status mk_pages_sync(mk_page_pool *pool, int32_t *page_table_dev, void *stream);
void mk_pages_destroy(mk_page_pool *pool);

/* Passage: none on the pages (error reporting of this library).
 * Synchronises `stream`, reads and clears the plan's device error word, and
 * returns the status it held.  It takes the stream the plan's steps run on
 * and an optional report (info, may be NULL) beyond the plain
 * mk_plan_last_error(plan) form: the stream says which work to wait for, and
 * the report names the site, CTA and offending value.  The read is one
 * copy on `stream` into host memory, then one synchronisation; clearing, when
 * an error was set, resets every control word of the plan. */
mk_status mk_plan_last_error(mk_plan *plan, void *stream, mk_device_error *info);

const char *mk_status_string(mk_status s);
const char *mk_error_site_string(int32_t site);

/* Passage: none on the pages.  Frees the plan's device memory.
 * Synchronises the device first. */
void mk_plan_destroy(mk_plan *plan);

/* ---------------------------------------------------------------------
 * Host-only introspection of the task graph (no GPU needed).
 * --------------------------------------------------------------------- */
typedef struct {
    int32_t cta;         /* worker CTA whose queue holds the task */
    int32_t op;          /* 1 QKV, 2 ATTN, 3 O, 4 GATE_UP, 5 DOWN, 6 LM_HEAD, 7 EMBED (batched only),
                            8 KV_APPEND (kv_append graphs only) */
    int32_t layer;
    int32_t wait_event;  /* -1: none */
    int32_t wait_count;  /* proceed when counter[wait_event] >= wait_count */
    int32_t signal_event;/* -1: none (attention: only the last split of a head signals) */
    int32_t a0, a1;      /* batch 1 projection: output rows [a0, a1);
                            batched projection: units [a0, a1), unit u = 128-row tile u / ceil(K/64),
                            64-column chunk u % ceil(K/64); embedding: items [a0, a1), item =
                            sequence * ceil(hidden/128) + 128-row tile; attention: batch row, kv head */
    int32_t a2, a3;      /* attention: split index, number of splits; projections: range number a2 */
} mk_task_info;

/* Passage: the task graph of "Compilar LLM en un MegaKernel…", "Parte 1.
 * Compilador" (tasks, events, dependencies), as a host-only listing.
 * Builds the task graph for `num_ctas` worker CTAs without touching a GPU.
 * Writes up to `capacity` tasks (queue order, CTA by CTA) to out, the task
 * count to *n_tasks and the number of event counters to *n_events.
 * MK_ERR_INVALID if capacity is too small (n_tasks still set). */
mk_status mk_plan_describe(const mk_model_cfg *cfg, const mk_plan_options *opt, int32_t num_ctas,
                           mk_task_info *out, int32_t capacity, int32_t *n_tasks, int32_t *n_events);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
