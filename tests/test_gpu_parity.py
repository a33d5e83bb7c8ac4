"""GPU parity: the megakernel (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Tolerances are the parity contract's: final logits
rel-L2 <= 1e-2 and max-abs <= 3e-2, greedy token equal whenever the oracle's
top-2 gap exceeds 0.05 (tests/harness.py)."""
import ctypes

import numpy as np
import pytest

import persistent_decode_megakernel_04_b300 as mk
import synth
from synth import WORKLOADS
from tests import harness

pytestmark = pytest.mark.gpu

TINY = WORKLOADS["tiny"].model


def _bits(t):
    import torch

    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_device_generator_matches_host_bit_for_bit(cuda_device):
    import torch

    for shape, tid, sig, off in [((4099,), 5, 0.02, 0.0), ((1000, 37), 17, 0.5, 0.0), ((513,), 3, 0.1, 1.0)]:
        t = torch.empty(shape, dtype=torch.bfloat16, device=cuda_device)
        synth._fill_device(t, 7, tid, sig, off)
        assert np.array_equal(_bits(t), synth.normal_bf16(shape, 7, tid, sig, off))
    # every tensor of the tiny model, and sampled rows of the 8B-shaped embedding
    dw, hw = synth.device_weights(TINY, 0), synth.host_weights(TINY, 0)
    assert np.array_equal(_bits(dw["embed"]), hw["embed"])
    for l in range(TINY.n_layers):
        for k in hw["layers"][l]:
            assert np.array_equal(_bits(dw["layers"][l][k]), hw["layers"][l][k]), (l, k)
    big = WORKLOADS["8b"].model
    t = torch.empty((64, big.hidden), dtype=torch.bfloat16, device=cuda_device)
    synth._fill_device(t, 0, synth.TID_EMBED, big.weight_std)
    assert np.array_equal(_bits(t), synth.normal_bf16((64, big.hidden), 0, synth.TID_EMBED, big.weight_std))


def test_device_kv_page_fill_matches_host(cuda_device):
    m = TINY
    kv = mk.KVCache(m, 2, 200, shuffle_seed=3)
    synth.device_kv_pages(kv.k[1], kv.page_table, m, 0, 1, "k", 2, kv.max_pages, 150, kv.page_size)
    ref = synth.host_kv(m, 0, 1, "k", 2, 150)
    pt = kv.page_table.cpu().numpy()
    pool = _bits(kv.k[1])
    for b in range(2):
        for t in (0, 63, 64, 149):
            assert np.array_equal(pool[pt[b, t // 64], :, t % 64, :], ref[b, t])


@pytest.mark.parametrize("gains", [False, True], ids=["unit-gains", "random-gains"])
def test_tiny_prompt_and_greedy_decode(cuda_device, gains):
    m = synth.with_random_gains(TINY) if gains else TINY
    wl = WORKLOADS["tiny"]
    max_seq = wl.seq_capacity
    plan, kv = harness.gpu_plan(m, max_seq)
    model = harness.oracle_model(m)
    prompt = synth.tokens(wl.prompt_len, 0, 0, m.vocab)
    stats = harness.run_teacher_forced(plan, kv, model, prompt, wl.decode_steps, max_seq)
    assert len(stats) == wl.decode_steps + 1


def test_tiny_ablation_matches_oracle(cuda_device):
    wl = WORKLOADS["tiny"]
    plan, kv = harness.gpu_plan(TINY, wl.seq_capacity)
    model = harness.oracle_model(TINY)
    prompt = synth.tokens(wl.prompt_len, 0, 1, TINY.vocab)
    harness.run_teacher_forced(plan, kv, model, prompt, 8, wl.seq_capacity, ablation_every=1)


def test_tiny_reduced_grid_and_permuted_schedule(cuda_device):
    # fewer worker CTAs than rows, odd split counts and a shuffled CTA assignment
    for opts in (mk.mk_plan_options(num_ctas=7, attn_splits=3, planner_seed=5),
                 mk.mk_plan_options(num_ctas=148, attn_splits=1, num_slots=2, slot_bytes=8192, planner_seed=9)):
        plan, kv = harness.gpu_plan(TINY, 128, opts=opts)
        model = harness.oracle_model(TINY)
        prompt = synth.tokens(70, 0, 2, TINY.vocab)  # crosses a KV page boundary
        harness.run_teacher_forced(plan, kv, model, prompt, 4, 128)


def test_host_buffer_entry_point_and_greedy_next(cuda_device):
    import torch

    wl = WORKLOADS["tiny"]
    plan, kv = harness.gpu_plan(TINY, wl.seq_capacity)
    prompt = synth.tokens(9, 0, 3, TINY.vocab)
    toks = torch.tensor(prompt, dtype=torch.int32, device=cuda_device).view(1, -1)
    logits = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
    plan.prefill(toks, kv, logits)
    nxt = torch.empty(1, dtype=torch.int32, device=cuda_device)
    pos = torch.full((1,), 8, dtype=torch.int32, device=cuda_device)
    plan.greedy_next(logits, nxt, pos)
    ref_tok = int(np.argmax(logits.cpu().numpy()[0]))
    assert int(nxt.item()) == ref_tok and int(pos.item()) == 9
    # the host-buffer call equals the device call at the same position
    host_logits = np.empty((1, TINY.vocab), dtype=np.float32)
    plan.decode_step_host(np.array([ref_tok], np.int32), np.array([9], np.int32), kv, host_logits)
    dev_logits = torch.empty_like(logits)
    plan.decode_step(nxt, pos, kv, dev_logits)
    plan.check()
    assert np.array_equal(host_logits, dev_logits.cpu().numpy())


def test_repeated_steps_are_bitwise_deterministic(cuda_device):
    import torch

    wl = WORKLOADS["tiny"]
    plan, kv = harness.gpu_plan(TINY, wl.seq_capacity)
    toks = torch.tensor(synth.tokens(20, 0, 4, TINY.vocab), dtype=torch.int32, device=cuda_device).view(1, -1)
    logits = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
    plan.prefill(toks, kv, logits)
    t = torch.tensor([5], dtype=torch.int32, device=cuda_device)
    p = torch.tensor([20], dtype=torch.int32, device=cuda_device)
    outs = []
    for _ in range(3):
        plan.decode_step(t, p, kv, logits)  # rewrites the same cache slot
        outs.append(logits.cpu().numpy().copy())
    plan.check()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_out_of_range_token_and_position_are_reported_not_faulted(cuda_device):
    import torch

    wl = WORKLOADS["tiny"]
    plan, kv = harness.gpu_plan(TINY, wl.seq_capacity)
    logits = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
    good_t = torch.tensor([3], dtype=torch.int32, device=cuda_device)
    good_p = torch.tensor([0], dtype=torch.int32, device=cuda_device)
    for tok, pos, site in ((TINY.vocab, 0, 6), (-1, 0, 6), (3, wl.seq_capacity, 7), (3, -5, 7)):
        t = torch.tensor([tok], dtype=torch.int32, device=cuda_device)
        p = torch.tensor([pos], dtype=torch.int32, device=cuda_device)
        plan.decode_step(t, p, kv, logits)
        info = plan.last_error()
        assert info.status == mk.MK_ERR_BOUNDS and info.site == site
        # the error was cleared by reading it: a valid step runs again
        plan.decode_step(good_t, good_p, kv, logits)
        assert plan.last_error().status == mk.MK_OK
    assert np.all(np.isfinite(logits.cpu().numpy()))


def test_bad_page_id_is_reported_not_faulted(cuda_device):
    import torch

    plan, kv = harness.gpu_plan(TINY, 128)
    logits = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
    kv.page_table[0, 1] = kv.num_pages  # one past the pool
    plan.decode_step(torch.tensor([3], dtype=torch.int32, device=cuda_device),
                     torch.tensor([70], dtype=torch.int32, device=cuda_device), kv, logits)
    info = plan.last_error()
    assert info.status == mk.MK_ERR_BOUNDS and info.site == 8 and info.detail == kv.num_pages


def test_unreachable_event_times_out_cleanly(cuda_device):
    import torch

    wl = WORKLOADS["tiny"]
    # waiters of layer 0's attention event need one more signal than exists
    opts = mk.mk_plan_options(timeout_ms=100, test_unreachable_event=2)
    plan, kv = harness.gpu_plan(TINY, wl.seq_capacity, opts=opts)
    logits = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
    t = torch.tensor([3], dtype=torch.int32, device=cuda_device)
    p = torch.tensor([0], dtype=torch.int32, device=cuda_device)
    plan.decode_step(t, p, kv, logits)
    info = plan.last_error()
    assert info.status == mk.MK_ERR_TIMEOUT and info.site == 1 and info.detail == 1
    # the context is intact: a normal plan on the same device still matches the oracle
    good, kv2 = harness.gpu_plan(TINY, wl.seq_capacity)
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced(good, kv2, model, synth.tokens(5, 0, 5, TINY.vocab), 2, wl.seq_capacity)


def test_invalid_kv_descriptor_rejected_on_host(cuda_device):
    import torch

    plan, kv = harness.gpu_plan(TINY, 128)
    logits = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
    t = torch.tensor([3], dtype=torch.int32, device=cuda_device)
    d = kv.desc
    bads = [mk.mk_kv_cache(d.k_pool, d.v_pool, d.page_table, d.num_pages, 1),  # 64 positions < max_seq 128
            mk.mk_kv_cache(d.k_pool + 2, d.v_pool, d.page_table, d.num_pages, d.max_pages_per_seq),  # misaligned
            mk.mk_kv_cache(d.k_pool, None, d.page_table, d.num_pages, d.max_pages_per_seq),
            mk.mk_kv_cache(d.k_pool, d.v_pool, d.page_table, 0, d.max_pages_per_seq)]
    for bad in bads:
        st = mk.lib().mk_decode_step(plan.h, t.data_ptr(), t.data_ptr(), ctypes.byref(bad), logits.data_ptr(),
                                     None)
        assert st == mk.MK_ERR_INVALID
    assert mk.lib().mk_decode_step(plan.h, t.data_ptr(), t.data_ptr(), ctypes.byref(d), None, None) == \
        mk.MK_ERR_INVALID


def test_tiny_long_prompt_through_decode_path(cuda_device):
    # 130-token prompt: several KV pages, splits that straddle pages; the
    # prompt runs through the decode step once per position
    plan, kv = harness.gpu_plan(TINY, 256, opts=mk.mk_plan_options(prefill_by_decode=1))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced(plan, kv, model, synth.tokens(130, 0, 6, TINY.vocab), 3, 256)


@pytest.mark.parametrize("T", [1, 7, 64, 65, 130, 200])
def test_chunked_prefill_matches_oracle_and_decode_prefill(cuda_device, T):
    """The chunked-prefill engine (up to 64 consecutive tokens of the
    sequence per launch on the tensor-core path, K/V appended before the
    rows attend to each other): the last position's logits match the oracle,
    and the K/V it leaves in the cache match the decode-step prefill's to
    bf16 rounding, so decode continues from it (a short last chunk, page
    crossings, a single token)."""
    import torch

    max_seq = 256
    plan, kv = harness.gpu_plan(TINY, max_seq)
    ref_plan, ref_kv = harness.gpu_plan(TINY, max_seq, opts=mk.mk_plan_options(prefill_by_decode=1))
    model = harness.oracle_model(TINY)
    prompt = synth.tokens(T, 0, 14, TINY.vocab)
    kc, vc = model.new_cache(max_seq)
    ref = model.prefill(kc, vc, prompt)
    toks = torch.tensor(prompt, dtype=torch.int32, device=cuda_device).view(1, -1)
    a = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
    b = torch.empty_like(a)
    plan.prefill(toks, kv, a)
    ref_plan.prefill(toks, ref_kv, b)
    plan.check()
    ref_plan.check()
    harness.compare_logits(a.cpu().numpy()[0], ref, f"chunked prefill of {T}")
    harness.compare_logits(a.cpu().numpy()[0], b.cpu().numpy()[0], f"chunked vs decode prefill of {T}")
    # the cache entries of every prompt position, gathered through each page table
    for pool, ref_pool in ((kv.k, ref_kv.k), (kv.v, ref_kv.v)):
        for t in range(T):
            pa = int(kv.page_table[0, t // 64])
            pb = int(ref_kv.page_table[0, t // 64])
            x = pool[:, pa, :, t % 64].float()
            y = ref_pool[:, pb, :, t % 64].float()
            assert torch.allclose(x, y, rtol=2 ** -7, atol=1e-3), f"cache position {t}"
    # decode continues from the chunked prefill's cache
    harness.run_teacher_forced(plan, kv, model, prompt, 3, max_seq)


def test_batched_kv_append_graph_decode(cuda_device):
    """Batched decode on the kv-append graph (each row's K/V appended by a
    task of its own, then read from the cache by attention) against the
    oracle."""
    from tests.test_gpu_batched import prompts

    max_seq = 128
    plan, kv = harness.gpu_plan(TINY, max_seq, batch=8, opts=mk.mk_plan_options(kv_append=1))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced_batch(plan, kv, model, prompts(8, 30, seed=4), 5, max_seq, rows=[0, 5, 7])


@pytest.mark.parametrize("name,ctx,steps", [("1b", 512, 3), ("8b", 39, 3), ("8b-batch", 4096, 2)])
def test_full_size_decode_from_seeded_cache(cuda_device, name, ctx, steps):
    """Full-size shapes in the launch configuration the bench times (every
    SM, default ring): decode steps at the workload's context length, from a
    seeded stand-in cache that both sides read."""
    wl = WORKLOADS[name]
    m = wl.model
    max_seq = ((ctx + steps + 64) // 64) * 64
    plan, kv = harness.gpu_plan(m, max_seq)
    model = harness.oracle_model(m)
    caches = harness.fill_synthetic_cache(kv, model, m, ctx, 1, max_seq)
    stats = harness.run_from_cache(plan, kv, model, caches, ctx, steps, synth.tokens(1, wl.seed, 0, m.vocab))
    print(name, stats)


@pytest.mark.parametrize("name,steps", [("8b", 16), ("1b", 8)])
def test_full_size_prompt_prefill_and_greedy_decode(cuda_device, name, steps):
    """The stated workloads end to end at full size, in the launch
    configuration the bench times (every SM, default ring): the 8B-shaped
    decoder's 39-token random prompt and the 1B-shaped decoder's 512-token
    random-ID context, prefilled through mk_prefill on the GPU and token by
    token by the oracle, then teacher-forced greedy decode steps, the logits
    compared at every step.  The cache holds the keys and values the model
    itself computed for the prompt, and the oracle's cache stores them as
    bf16, as the paged bf16 cache does: on these random-init decoders the
    rounding alone moves the fp64 oracle's own logits by 1.8e-2 rel-L2 after
    the 8B prompt, beyond the tolerance, so an fp64 cache would measure the
    cache's storage type, not the kernels."""
    wl = WORKLOADS[name]
    m = wl.model
    max_seq = ((wl.prompt_len + steps + 8 + 63) // 64) * 64
    plan, kv = harness.gpu_plan(m, max_seq)
    model = harness.oracle_model(m, kv_bf16=True)
    prompt = synth.tokens(wl.prompt_len, wl.seed, 0, m.vocab)
    stats = harness.run_teacher_forced(plan, kv, model, prompt, steps, max_seq)
    assert len(stats) == steps + 1
    print(name, "rel-L2", [round(x["rel_l2"], 5) for x in stats], "max-abs", [round(x["max_abs"], 4) for x in stats])


@pytest.mark.parametrize("m", [synth.TINY_G8, synth.TINY_MHA, synth.TINY_D128], ids=["g8", "mha", "d128"])
def test_tiny_variants_group_sizes_and_head_dim(cuda_device, m):
    """GQA groups of 8 and 1 (two and one MMA column tiles in attention) and
    head_dim 128 (two swizzled K/V halves), prompt crossing a KV page."""
    plan, kv = harness.gpu_plan(m, 128)
    model = harness.oracle_model(m)
    harness.run_teacher_forced(plan, kv, model, synth.tokens(70, 0, 8, m.vocab), 4, 128)


@pytest.mark.parametrize("opts", [dict(max_inflight=1, attn_splits=1),
                                  dict(max_inflight=6, attn_splits=2, l2_prefetch_kb=256),
                                  dict(num_slots=3, slot_bytes=8192, attn_splits=1)],
                         ids=["inflight1", "uncapped-prefetch", "no-two-block-steps"])
def test_tiny_ring_and_attention_step_options(cuda_device, opts):
    """Ring copies capped at one in flight or uncapped, the optional L2
    prefetch, and attention taking both two-block and one-block steps (three
    cached blocks in one split; one and two blocks in two splits), or only
    one-block steps when the ring cannot hold two blocks at once."""
    plan, kv = harness.gpu_plan(TINY, 256, opts=mk.mk_plan_options(**opts))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced(plan, kv, model, synth.tokens(150, 0, 9, TINY.vocab), 4, 256)


@pytest.mark.parametrize("name,batch", [("tiny", 1), ("1b", 1), ("tiny", 4), ("tiny", 24), ("tiny", 64)],
                         ids=["tiny-b1", "1b-b1", "tiny-b4", "tiny-b24", "tiny-b64"])
def test_fused_greedy_step_matches_step_then_pick(cuda_device, name, batch):
    """mk_decode_step_greedy (the pick fused into the decode launch: the LM
    head's matvec rows at batch 1, its tensor-core tile epilogue when
    batched) gives the logits, tokens and positions of mk_decode_step
    followed by mk_greedy_next, bit for bit."""
    import torch

    m = WORKLOADS[name].model
    max_seq = 128
    plan, kv_a = harness.gpu_plan(m, max_seq, batch=batch)
    kv_b = mk.KVCache(m, batch, max_seq, shuffle_seed=1)
    prompt = np.stack([synth.tokens(40, 0, b, m.vocab) for b in range(batch)])
    logits_a = torch.empty((batch, m.vocab), dtype=torch.float32, device=cuda_device)
    plan.prefill(torch.tensor(prompt, dtype=torch.int32, device=cuda_device), kv_a, logits_a)
    plan.check()
    kv_b.k.copy_(kv_a.k)
    kv_b.v.copy_(kv_a.v)
    kv_b.page_table.copy_(kv_a.page_table)
    tok_a = torch.zeros(batch, dtype=torch.int32, device=cuda_device)
    pos_a = torch.full((batch,), 39, dtype=torch.int32, device=cuda_device)
    plan.greedy_next(logits_a, tok_a, pos_a)
    tok_b, pos_b = tok_a.clone(), pos_a.clone()
    logits_b = torch.empty_like(logits_a)
    for step in range(4):
        plan.decode_step(tok_a, pos_a, kv_a, logits_a)
        plan.greedy_next(logits_a, tok_a, pos_a)
        plan.decode_step_greedy(tok_b, pos_b, kv_b, logits_b)
        plan.check()
        assert torch.equal(logits_a, logits_b), f"step {step}: logits differ"
        assert torch.equal(tok_a, tok_b) and torch.equal(pos_a, pos_b), f"step {step}: {tok_a} {tok_b} {pos_a} {pos_b}"
        assert int(pos_b[0]) == 41 + step
    # the host-buffer form from the same state: its picks are the device form's
    kv_b.k.copy_(kv_a.k)
    kv_b.v.copy_(kv_a.v)
    h_tok = tok_a.cpu().numpy().copy()
    h_pos = pos_a.cpu().numpy().copy()
    h_nxt = np.zeros(batch, np.int32)
    for step in range(3):
        plan.decode_step_greedy(tok_a, pos_a, kv_a, logits_a)
        plan.decode_step_greedy_host(h_tok, h_pos, kv_b, h_nxt)
        plan.check()
        assert np.array_equal(h_nxt, tok_a.cpu().numpy()), f"host step {step}: {h_nxt} {tok_a}"
        h_tok[:] = h_nxt
        h_pos += 1
        assert np.array_equal(h_pos, pos_a.cpu().numpy())


@pytest.mark.parametrize("batch", [1, 8])
def test_fused_greedy_pick_equals_oracle_argmax(cuda_device, batch):
    """The token the fused pick writes is the oracle's greedy token wherever
    the oracle's top-2 logit gap exceeds 0.05 (teacher forcing: every step
    starts from the oracle's token).  The tiny decoder with weights
    N(0, 0.06) spreads its logits enough (std about 1) that most steps have
    such a gap."""
    from dataclasses import replace

    import torch

    m = replace(WORKLOADS["tiny"].model, weight_std=0.06, name="tiny-std0.06")
    max_seq, T, steps = 128, 24, 8
    plan, kv = harness.gpu_plan(m, max_seq, batch=batch)
    model = harness.oracle_model(m)
    prompts = np.stack([synth.tokens(T, 0, 200 + b, m.vocab) for b in range(batch)])
    caches = [model.new_cache(max_seq) for _ in range(batch)]
    refs = [model.prefill(caches[b][0], caches[b][1], prompts[b]) for b in range(batch)]
    logits = torch.empty((batch, m.vocab), dtype=torch.float32, device=cuda_device)
    plan.prefill(torch.tensor(prompts, dtype=torch.int32, device=cuda_device), kv, logits)
    plan.check()
    checked = 0
    for i in range(steps):
        pos = T + i
        forced = [int(np.argmax(r)) for r in refs]
        refs = [model.decode_step(caches[b][0], caches[b][1], forced[b], pos) for b in range(batch)]
        tok = torch.tensor(forced, dtype=torch.int32, device=cuda_device)
        pos_d = torch.full((batch,), pos, dtype=torch.int32, device=cuda_device)
        plan.decode_step_greedy(tok, pos_d, kv, logits)
        plan.check()
        got = tok.cpu().numpy()
        assert np.all(pos_d.cpu().numpy() == pos + 1)
        for b in range(batch):
            top2 = np.sort(refs[b])[-2:]
            if top2[1] - top2[0] > harness.ARGMAX_GAP:
                assert int(got[b]) == int(np.argmax(refs[b])), f"step {i} row {b}"
                checked += 1
    assert checked >= steps * batch // 2


@pytest.mark.parametrize("m", [synth.TINY_WIDE, synth.TINY_LONGFF, synth.TINY_FFN6K],
                         ids=["wide-hidden", "wide-ffn", "ffn-6144-tma"])
@pytest.mark.parametrize("opts", [None, dict(num_ctas=7, attn_splits=3), dict(num_ctas=2, attn_splits=1)],
                         ids=["all-sms", "7ctas", "2ctas"])
def test_tiny_long_matvec_inputs(cuda_device, m, opts):
    """Batch-1 projections whose input is longer than the 4096 columns kept
    in registers stream the input from L2 piece by piece, with row groups
    taken several at a time: QKV, gate/up and the LM head of a 4608-wide
    hidden size (a ragged last piece, groups cut at the q/k/v boundaries) and
    the down projection of a 5000-wide feed-forward (one bulk copy per row
    and piece) and of a 6144-wide one (one 3-D TMA copy per slot, row groups
    cut short at the CTA's range end).  Two CTAs hold 512 or more rows each,
    so the per-group totals are flushed mid-task."""
    plan, kv = harness.gpu_plan(m, 128, opts=mk.mk_plan_options(**opts) if opts else None)
    model = harness.oracle_model(m)
    harness.run_teacher_forced(plan, kv, model, synth.tokens(24, 0, 13, m.vocab), 4, 128)


@pytest.mark.parametrize("opts", [dict(jit=1), dict(jit=4), dict(jit=2, num_ctas=7, attn_splits=3),
                                  dict(jit=1, num_ctas=1, attn_splits=2)],
                         ids=["jit1", "jit4", "jit2-7ctas", "jit1-1cta"])
def test_dynamic_dispatch_matches_oracle(cuda_device, opts):
    """Dynamic dispatch (tasks claimed by the CTAs at run time, stage by
    stage) computes the same decoder: prompt and teacher-forced decode steps
    against the oracle, with fine ranges, a reduced grid and a single CTA
    that claims every task."""
    import torch

    plan, kv = harness.gpu_plan(TINY, 256, opts=mk.mk_plan_options(**opts))
    model = harness.oracle_model(TINY)
    harness.run_teacher_forced(plan, kv, model, synth.tokens(70, 0, 15, TINY.vocab), 5, 256)
    t = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    logits = torch.empty((1, TINY.vocab), dtype=torch.float32, device=cuda_device)
    st = mk.lib().mk_decode_step_ablation(plan.h, t.data_ptr(), t.data_ptr(), ctypes.byref(kv.desc),
                                          logits.data_ptr(), None)
    assert st == mk.MK_ERR_UNSUPPORTED  # one operator per launch needs the static queues


def test_dynamic_dispatch_full_size_from_seeded_cache(cuda_device):
    """The 8B-shaped decoder under dynamic dispatch, from a seeded cache."""
    wl = WORKLOADS["8b"]
    m = wl.model
    ctx, steps = 100, 2
    max_seq = ((ctx + steps + 64) // 64) * 64
    plan, kv = harness.gpu_plan(m, max_seq, opts=mk.mk_plan_options(jit=1))
    model = harness.oracle_model(m)
    caches = harness.fill_synthetic_cache(kv, model, m, ctx, 1, max_seq)
    harness.run_from_cache(plan, kv, model, caches, ctx, steps, synth.tokens(1, wl.seed, 0, m.vocab))


@pytest.mark.parametrize("m", [WORKLOADS["tiny"].model, synth.TINY_MHA, synth.TINY_D128, synth.TINY_G8],
                         ids=["g2", "mha", "d128-g4", "g8"])
@pytest.mark.parametrize("batch", [1, 3])
def test_long_splits_warp_local_attention(cuda_device, m, batch):
    """Splits of four or more cached blocks run attention warp by warp (each
    warp its own tokens: scores, online softmax and value sums in registers,
    then a tree merge of the warps); one split per head over a 300-token
    prompt (five blocks: two two-block steps and a one-block step) for GQA
    groups of 2, 1 and 4 (head_dim 128), and 8, which keeps the per-block
    path."""
    from tests.test_gpu_batched import prompts

    max_seq = 384
    plan, kv = harness.gpu_plan(m, max_seq, batch=batch, opts=mk.mk_plan_options(attn_splits=1))
    model = harness.oracle_model(m)
    if batch == 1:
        harness.run_teacher_forced(plan, kv, model, synth.tokens(300, 0, 16, m.vocab), 4, max_seq)
    else:
        harness.run_teacher_forced_batch(plan, kv, model, prompts(batch, 300, seed=11, vocab=m.vocab), 3, max_seq,
                                         rows=[0, batch - 1])


@pytest.mark.parametrize("case", [dict(batch=1), dict(batch=1, prefill_by_decode=1), dict(batch=1, tensor_cores=1),
                                  dict(batch=24), dict(batch=6, jit=1)],
                         ids=["b1", "b1-decode-prefill", "b1-tc", "b24", "b6-jit"])
def test_poisoned_scratch_is_never_read_unwritten(cuda_device, case):
    """Every activation buffer of the plan's scratch is NaN-filled before each
    step (test_poison_scratch): the prompt prefill (chunked engine, or decode
    steps), teacher-forced decode steps and launch-per-operator steps must
    still match the oracle, so no step reads a scratch value it did not write
    in that step."""
    m = TINY
    B = case.pop("batch")
    max_seq = 128
    plan, kv = harness.gpu_plan(m, max_seq, batch=B, opts=mk.mk_plan_options(test_poison_scratch=1, **case))
    model = harness.oracle_model(m)
    prompts = np.stack([synth.tokens(21, 4, 400 + b, m.vocab) for b in range(B)])
    rows = sorted({0, B - 1})
    harness.run_teacher_forced_batch(plan, kv, model, prompts, 4, max_seq, rows=rows,
                                     ablation_every=0 if case.get("jit") else 3)
