"""GPU parity of the batched decode path (tcgen05 tensor-core projections,
fused epilogues, stream-K row tiles) against the fp64 oracle, through the C
ABI.  Same tolerances as the batch-1 path (tests/harness.py)."""
import numpy as np
import pytest

import persistent_decode_megakernel_04_b300 as mk
import synth
from synth import WORKLOADS
from tests import harness

pytestmark = pytest.mark.gpu

TINY = WORKLOADS["tiny"].model


def prompts(B, T, seed=0, vocab=TINY.vocab):
    return np.stack([synth.tokens(T, seed, 100 + b, vocab) for b in range(B)])


@pytest.mark.parametrize("B", [2, 16, 24, 64])
def test_tiny_batched_prompt_and_decode(cuda_device, B):
    # B=24 pads the MMA N to 32 (rows 24..31 of the activation tiles read as zero)
    max_seq = 128
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=B)
    model = harness.oracle_model(TINY)
    rows = sorted({0, 1, B // 2, B - 1})
    harness.run_teacher_forced_batch(plan, kv, model, prompts(B, 20), 6, max_seq, rows=rows)


def test_tiny_batched_random_gains_and_ablation(cuda_device):
    m = synth.with_random_gains(TINY)
    max_seq = 128
    plan, kv = harness.gpu_plan(m, max_seq, batch=8)
    model = harness.oracle_model(m)
    harness.run_teacher_forced_batch(plan, kv, model, prompts(8, 12, seed=3), 4, max_seq, rows=[0, 3, 7],
                                     ablation_every=2)


@pytest.mark.parametrize("opts", [dict(num_ctas=7, attn_splits=3, planner_seed=5),
                                  dict(num_ctas=148, attn_splits=1, num_slots=3, planner_seed=9),
                                  dict(num_ctas=1), dict(tc_tile_split=1), dict(tc_tile_split=2, planner_seed=3),
                                  dict(tc_tile_split=3, num_ctas=20), dict(num_ctas=5)],
                         ids=["7ctas", "3slots", "1cta", "split1", "split2", "split3-20ctas", "5ctas-balanced-splits"])
def test_tiny_batched_schedules(cuda_device, opts):
    # row tiles shared by several ranges (fixup), a permuted CTA assignment,
    # a shallow weight ring and a single worker CTA
    max_seq = 128
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=4, opts=mk.mk_plan_options(**opts))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced_batch(plan, kv, model, prompts(4, 70, seed=2), 3, max_seq, rows=[0, 3])


def test_tiny_batched_ragged_positions(cuda_device):
    B, max_seq = 6, 256
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=B)
    model = harness.oracle_model(TINY)
    ctx = 150
    caches = harness.fill_synthetic_cache(kv, model, TINY, ctx, B, max_seq, rows=(0, 2, 5))
    ctxs = [ctx - 37 * b % 140 for b in range(B)]  # every row at its own position
    harness.run_from_cache_ragged(plan, kv, model, caches, ctxs, 3, synth.tokens(B, 0, 9, TINY.vocab), B)


def test_batched_rows_equal_single_sequence_runs(cuda_device):
    """Row b of a batched step equals the same sequence run alone (batch 1
    path) to within the parity tolerance."""
    import torch

    B, T, max_seq = 4, 16, 64
    P = prompts(B, T, seed=7)
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=B)
    logits = torch.empty((B, TINY.vocab), dtype=torch.float32, device=cuda_device)
    plan.prefill(torch.tensor(P, dtype=torch.int32, device=cuda_device), kv, logits)
    plan.check()
    got = logits.cpu().numpy()
    for b in range(B):
        p1, kv1 = harness.gpu_plan(TINY, max_seq, batch=1)
        l1 = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
        p1.prefill(torch.tensor(P[b:b + 1], dtype=torch.int32, device=cuda_device), kv1, l1)
        p1.check()
        harness.compare_logits(got[b], l1.cpu().numpy()[0], f"row {b} vs batch-1 run")


@pytest.mark.parametrize("B,split", [(8, 0), (32, 0), (64, 0), (64, 2)], ids=["8", "32", "64", "64-split2"])
def test_8b_batched_decode_from_seeded_cache(cuda_device, B, split):
    """The 8B-shaped decoder at 4096 cached tokens per sequence (paged,
    shuffled pages), in the launch configuration the bench times; the oracle
    checks rows 0 and B-1."""
    wl = WORKLOADS["8b-batch"]
    m = wl.model
    ctx, steps = 4096, 2
    max_seq = ((ctx + steps + 64) // 64) * 64
    plan, kv = harness.gpu_plan(m, max_seq, batch=B, opts=mk.mk_plan_options(tc_tile_split=split))
    model = harness.oracle_model(m)
    caches = harness.fill_synthetic_cache(kv, model, m, ctx, B, max_seq, rows=(0, B - 1))
    harness.run_from_cache(plan, kv, model, caches, ctx, steps, synth.tokens(B, wl.seed, 0, m.vocab), batch=B)


def test_tiny_batch1_on_tensor_cores(cuda_device):
    """Batch 1 with the projections forced onto the tcgen05 path (N padded to
    16): the same task graph as the batched plans, one live row."""
    max_seq = 128
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=1, opts=mk.mk_plan_options(tensor_cores=1))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced_batch(plan, kv, model, prompts(1, 20, seed=5), 5, max_seq)


@pytest.mark.parametrize("m", [synth.TINY_G8, synth.TINY_MHA, synth.TINY_D128], ids=["g8", "mha", "d128"])
def test_tiny_variants_batched(cuda_device, m):
    max_seq = 128
    plan, kv = harness.gpu_plan(m, max_seq, batch=6)
    model = harness.oracle_model(m)
    harness.run_teacher_forced_batch(plan, kv, model, prompts(6, 66, seed=9, vocab=m.vocab), 3, max_seq,
                                     rows=[0, 5])


def test_70b_batched_first_decode_step(cuda_device):
    """The 70B-shaped decoder on one B300 (141 GB of bf16 weights, batch 16,
    2048 cached tokens per sequence): the first decode step from a seeded
    cache, checked by the oracle on rows 0 and 15.  The oracle regenerates
    each layer's weights on the host and discards them."""
    import torch

    import oracle

    torch.cuda.empty_cache()
    wl = WORKLOADS["70b"]
    m, B, ctx = wl.model, wl.batch, wl.prompt_len
    max_seq = ((ctx + 1 + 63) // 64) * 64
    plan, kv = harness.gpu_plan(m, max_seq, batch=B)
    for l in range(m.n_layers):
        for which, pool in (("k", kv.k), ("v", kv.v)):
            synth.device_kv_pages(pool[l], kv.page_table, m, wl.seed, l, which, B, kv.max_pages, ctx, kv.page_size)
    toks = synth.tokens(B, wl.seed, 0, m.vocab)
    logits = torch.empty((B, m.vocab), dtype=torch.float32, device=cuda_device)
    plan.decode_step(torch.tensor(toks, device=cuda_device), torch.full((B,), ctx, dtype=torch.int32,
                                                                       device=cuda_device), kv, logits)
    plan.check()
    got = logits.cpu().numpy()
    plan.close()
    del plan, kv
    torch.cuda.empty_cache()

    emb = synth.normal_bf16((m.vocab, m.hidden), wl.seed, synth.TID_EMBED, m.weight_std)
    lm = synth.normal_bf16((m.vocab, m.hidden), wl.seed, synth.TID_LM_HEAD, m.weight_std)
    fin = synth.normal_bf16((m.hidden,), wl.seed, synth.TID_FINAL_NORM, 0.0, 1.0)
    model = oracle.Model(m, {"embed": emb, "lm_head": lm, "final_norm": fin})
    rows = (0, B - 1)
    xs = {b: model.embed_token(int(toks[b])) for b in rows}
    for l in range(m.n_layers):
        lw = synth.host_layer_weights(m, wl.seed, l)
        kh = synth.host_kv(m, wl.seed, l, "k", B, ctx)
        vh = synth.host_kv(m, wl.seed, l, "v", B, ctx)
        for b in rows:
            kc = np.zeros((max_seq, m.n_kv_heads, m.head_dim))
            vc = np.zeros_like(kc)
            kc[:ctx] = synth.bf16_to_f64(kh[b])
            vc[:ctx] = synth.bf16_to_f64(vh[b])
            model.layer_step(lw, kc, vc, ctx, xs[b])
    for b in rows:
        harness.compare_logits(got[b], model.head(xs[b]), f"70B row {b}")


def test_continuous_batching_admits_grows_and_retires_sequences(cuda_device):
    """Continuous batching on a 4-row plan over a 10-page pool: sequences are
    admitted into free rows (prompt prefilled into the row's own pages by
    mk_prefill_row), decode with their own positions, grow page by page
    (one crosses a page boundary mid-run), retire, and a later sequence
    reuses the freed pages; a row never admitted runs on the scratch page.
    Every live row's logits match the oracle at every step (teacher
    forcing: each is fed the oracle's greedy token)."""
    import torch

    m = TINY
    B, max_seq, page = 4, 256, 64
    plan, _ = harness.gpu_plan(m, max_seq, batch=B)
    kv = mk.KVCache(m, B, max_seq, num_pages=10)
    pool = mk.PagePool(10, B, kv.max_pages, page)
    model = harness.oracle_model(m)
    live = {}  # row -> [oracle k cache, v cache, position, next token]
    V = m.vocab

    def admit(row, T, seq):
        prompt = synth.tokens(T, 0, 300 + seq, V)
        assert pool.admit(row, T) == mk.MK_OK
        pool.sync(kv.page_table)
        kc, vc = model.new_cache(max_seq)
        ref = model.prefill(kc, vc, prompt)
        out = torch.empty(V, dtype=torch.float32, device=cuda_device)
        plan.prefill_row(row, torch.tensor(prompt, dtype=torch.int32, device=cuda_device), kv, out)
        plan.check()
        harness.compare_logits(out.cpu().numpy(), ref, f"prefill of row {row}")
        live[row] = [kc, vc, T, int(np.argmax(ref))]

    def step(i):
        for row, st in live.items():
            assert pool.extend(row, st[2] + 1) == mk.MK_OK
        pool.sync(kv.page_table)
        tok = np.zeros(B, np.int32)
        pos = np.zeros(B, np.int32)
        refs = {}
        for row, st in live.items():
            tok[row], pos[row] = st[3], st[2]
            refs[row] = model.decode_step(st[0], st[1], st[3], st[2])
        logits = torch.empty((B, V), dtype=torch.float32, device=cuda_device)
        plan.decode_step(torch.tensor(tok, device=cuda_device), torch.tensor(pos, device=cuda_device), kv, logits)
        plan.check()
        got = logits.cpu().numpy()
        for row, ref in refs.items():
            harness.compare_logits(got[row], ref, f"step {i} row {row} (pos {pos[row]})")
            live[row][2] += 1
            live[row][3] = int(np.argmax(ref))

    admit(0, 20, 0)
    admit(2, 125, 1)  # crosses its second page boundary at position 128
    for i in range(6):
        step(i)
    assert live[2][2] == 131 and pool.table()[2, 2] != pool.scratch_page
    free_before = pool.free_count
    assert pool.retire(0) == mk.MK_OK and pool.free_count == free_before + 1
    del live[0]
    admit(0, 33, 2)  # reuses the retired sequence's page
    for i in range(6, 9):
        step(i)
    admit(3, 5, 3)
    for i in range(9, 12):
        step(i)
    assert np.all(pool.table()[1] == pool.scratch_page)  # row 1 never admitted
    pool.close()


def test_tiny_batched_dynamic_dispatch(cuda_device):
    """Batched (tensor-core) plan under dynamic dispatch against the oracle."""
    max_seq = 128
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=8, opts=mk.mk_plan_options(jit=1))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced_batch(plan, kv, model, prompts(8, 40, seed=6), 4, max_seq, rows=[0, 3, 7])


@pytest.mark.parametrize("B,sub", [(8, 1), (64, 1), (24, 2)], ids=["b8-sub1", "b64-sub1", "b24-sub2"])
def test_tiny_batched_k_subtiles(cuda_device, B, sub):
    """Projection units of one or two 64-column K sub-tiles (tc_k_subtiles),
    against the default for the batch; the tiny decoder's FFN width 688 is
    not a multiple of 128, so the last unit's second sub-tile reads past K
    (zero-filled on both operands)."""
    max_seq = 128
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=B, opts=mk.mk_plan_options(tc_k_subtiles=sub))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced_batch(plan, kv, model, prompts(B, 20, seed=11), 4, max_seq, rows=[0, B - 1],
                                     ablation_every=2)


@pytest.mark.parametrize("B,opts", [(64, {}), (8, dict(jit=1)), (1, {}), (40, dict(num_ctas=37))],
                         ids=["b64", "b8-jit", "b1", "b40-37ctas"])
def test_long_runs_with_poisoned_scratch(cuda_device, B, opts):
    """150 teacher-forced steps with every activation buffer NaN-filled
    before each step: a read racing ahead of its producer, or a ring slot
    reused a round early, would show as a parity failure somewhere along the
    run (the contexts grow across three 64-token pages)."""
    max_seq = 256
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=B,
                                opts=mk.mk_plan_options(test_poison_scratch=1, **opts))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced_batch(plan, kv, model, prompts(B, 20, seed=7), 150, max_seq, rows=sorted({0, B - 1}),
                                     ablation_every=0 if opts.get("jit") else 50)
