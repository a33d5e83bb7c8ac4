"""Shared set-up of GPU-vs-oracle parity runs (test infrastructure).

Both sides get the same seeded inputs from ``synth``: the GPU weights are
filled on the device, the oracle's on the host, by two independent
implementations of one generator (checked bit for bit in test_gpu_parity).
Nothing here feeds a GPU result into the oracle.
"""
from __future__ import annotations

import numpy as np

import oracle
import persistent_decode_megakernel_04_b300 as mk
import synth

# tolerances of the parity contract (final logits, fp32 GPU vs fp64 oracle)
REL_L2 = 1e-2
MAX_ABS = 3e-2
ARGMAX_GAP = 0.05


def compare_logits(gpu: np.ndarray, ref: np.ndarray, what: str) -> dict:
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU logits"
    rel = float(np.linalg.norm(gpu - ref) / np.linalg.norm(ref))
    mx = float(np.max(np.abs(gpu - ref)))
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS, f"{what}: max-abs {mx:.3e} > {MAX_ABS}"
    top2 = np.sort(ref)[-2:]
    gap = float(top2[1] - top2[0])
    if gap > ARGMAX_GAP:
        assert int(np.argmax(gpu)) == int(np.argmax(ref)), f"{what}: argmax differs with top-2 gap {gap:.3f}"
    return {"rel_l2": rel, "max_abs": mx, "gap": gap}


def gpu_plan(m, max_seq: int, batch: int = 1, seed: int = 0, opts=None, kv_shuffle: int | None = 1):
    import torch

    w = synth.device_weights(m, seed)
    torch.cuda.synchronize()
    plan = mk.Plan(m, w, batch=batch, max_seq=max_seq, opts=opts)
    kv = mk.KVCache(m, batch, max_seq, shuffle_seed=kv_shuffle)
    return plan, kv


_MODELS: dict = {}


def oracle_model(m, seed: int = 0, kv_bf16: bool = False) -> oracle.Model:
    """Host weights are generated once per (shape, seed) and kept (the
    8B-shaped ones take 16 GB).  kv_bf16: the oracle's cache stores its keys
    and values rounded to bf16, as the GPU's paged cache does."""
    key = (m, seed)
    if key not in _MODELS:
        if len(_MODELS) >= 2:
            _MODELS.pop(next(iter(_MODELS)))
        _MODELS[key] = synth.host_weights(m, seed)
    return oracle.Model(m, _MODELS[key], kv_bf16=kv_bf16)


def run_teacher_forced(plan: mk.Plan, kv: mk.KVCache, model: oracle.Model, prompt: np.ndarray, steps: int,
                       max_seq: int, ablation_every: int = 0):
    """Prefill `prompt` on both sides, then `steps` decode steps in which both
    are fed the ORACLE's greedy token.  Compares logits at every step."""
    import torch

    dev = torch.device("cuda")
    V = model.cfg.vocab
    stats = []
    kc, vc = model.new_cache(max_seq)
    ref = model.prefill(kc, vc, prompt)
    toks = torch.tensor(prompt, dtype=torch.int32, device=dev).view(1, -1)
    logits = torch.empty((1, V), dtype=torch.float32, device=dev)
    plan.prefill(toks, kv, logits)
    plan.check()
    stats.append(compare_logits(logits.cpu().numpy(), ref, "prefill"))
    pos = len(prompt)
    tok_d = torch.empty(1, dtype=torch.int32, device=dev)
    pos_d = torch.empty(1, dtype=torch.int32, device=dev)
    for i in range(steps):
        nxt = int(np.argmax(ref))
        ref = model.decode_step(kc, vc, nxt, pos)
        tok_d.fill_(nxt)
        pos_d.fill_(pos)
        if ablation_every and i % ablation_every == 0:
            plan.decode_step_ablation(tok_d, pos_d, kv, logits)
        else:
            plan.decode_step(tok_d, pos_d, kv, logits)
        plan.check()
        stats.append(compare_logits(logits.cpu().numpy(), ref, f"decode step {i} (pos {pos})"))
        pos += 1
    return stats


def fill_synthetic_cache(plan_kv: mk.KVCache, model: oracle.Model, m, ctx: int, batch: int, max_seq: int,
                         seed: int = 0, rows=(0,)):
    """Seeded stand-in contents for cache positions [0, ctx): written into the
    GPU pages by the device generator and into the oracle's caches (one per
    checked batch row) by the host generator."""
    caches = {b: model.new_cache(max_seq) for b in rows}
    for l in range(m.n_layers):
        for which, pool in (("k", plan_kv.k), ("v", plan_kv.v)):
            synth.device_kv_pages(pool[l], plan_kv.page_table, m, seed, l, which, batch, plan_kv.max_pages, ctx,
                                  plan_kv.page_size)
            host = synth.host_kv(m, seed, l, which, batch, ctx)
            for b in rows:
                dst = caches[b][0 if which == "k" else 1]
                dst[l, :ctx] = synth.bf16_to_f64(host[b])
    return caches


def run_from_cache(plan: mk.Plan, kv: mk.KVCache, model: oracle.Model, caches: dict, ctx: int, steps: int,
                   first_tokens, batch: int = 1):
    """Decode steps at positions ctx, ctx+1, ... from a filled cache; every
    checked row is fed the oracle's greedy token (teacher forcing)."""
    import torch

    dev = torch.device("cuda")
    V = model.cfg.vocab
    tok_h = np.array(first_tokens, dtype=np.int32)
    logits = torch.empty((batch, V), dtype=torch.float32, device=dev)
    stats = []
    for i in range(steps):
        pos = ctx + i
        refs = {b: model.decode_step(caches[b][0], caches[b][1], int(tok_h[b]), pos) for b in caches}
        plan.decode_step(torch.tensor(tok_h, device=dev), torch.full((batch,), pos, dtype=torch.int32, device=dev),
                         kv, logits)
        plan.check()
        got = logits.cpu().numpy()
        for b, ref in refs.items():
            stats.append(compare_logits(got[b], ref, f"row {b} step {i} (pos {pos})"))
            tok_h[b] = int(np.argmax(ref))
    return stats


def run_teacher_forced_batch(plan: mk.Plan, kv: mk.KVCache, model: oracle.Model, prompts: np.ndarray, steps: int,
                             max_seq: int, rows=None, ablation_every: int = 0):
    """Batched form of run_teacher_forced: prompts [B][T] are prefilled
    together; every decode step feeds each checked row the ORACLE's greedy
    token (unchecked rows follow the GPU's own greedy token).  Compares the
    checked rows' logits at every step."""
    import torch

    dev = torch.device("cuda")
    B, T = prompts.shape
    V = model.cfg.vocab
    rows = list(range(B)) if rows is None else list(rows)
    caches = {b: model.new_cache(max_seq) for b in rows}
    refs = {b: model.prefill(caches[b][0], caches[b][1], prompts[b]) for b in rows}
    logits = torch.empty((B, V), dtype=torch.float32, device=dev)
    plan.prefill(torch.tensor(prompts, dtype=torch.int32, device=dev), kv, logits)
    plan.check()
    got = logits.cpu().numpy()
    stats = [compare_logits(got[b], refs[b], f"prefill row {b}") for b in rows]
    tok = np.argmax(got, axis=1).astype(np.int32)
    for i in range(steps):
        pos = T + i
        for b in rows:
            tok[b] = int(np.argmax(refs[b]))
            refs[b] = model.decode_step(caches[b][0], caches[b][1], int(tok[b]), pos)
        tok_d = torch.tensor(tok, device=dev)
        pos_d = torch.full((B,), pos, dtype=torch.int32, device=dev)
        if ablation_every and i % ablation_every == 0:
            plan.decode_step_ablation(tok_d, pos_d, kv, logits)
        else:
            plan.decode_step(tok_d, pos_d, kv, logits)
        plan.check()
        got = logits.cpu().numpy()
        stats += [compare_logits(got[b], refs[b], f"row {b} decode step {i} (pos {pos})") for b in rows]
        tok = np.argmax(got, axis=1).astype(np.int32)
    return stats


def run_from_cache_ragged(plan: mk.Plan, kv: mk.KVCache, model: oracle.Model, caches: dict, ctxs, steps: int,
                          first_tokens, batch: int):
    """Decode steps from a seeded cache where row b starts at its own
    position ctxs[b] (ragged contexts).  Checked rows (the keys of `caches`)
    are teacher-forced with the oracle's greedy token."""
    import torch

    dev = torch.device("cuda")
    V = model.cfg.vocab
    tok_h = np.array(first_tokens, dtype=np.int32)
    pos_h = np.array(ctxs, dtype=np.int32)
    logits = torch.empty((batch, V), dtype=torch.float32, device=dev)
    stats = []
    for i in range(steps):
        refs = {b: model.decode_step(caches[b][0], caches[b][1], int(tok_h[b]), int(pos_h[b])) for b in caches}
        plan.decode_step(torch.tensor(tok_h, device=dev), torch.tensor(pos_h, device=dev), kv, logits)
        plan.check()
        got = logits.cpu().numpy()
        for b, ref in refs.items():
            stats.append(compare_logits(got[b], ref, f"row {b} step {i} (pos {pos_h[b]})"))
            tok_h[b] = int(np.argmax(ref))
        for b in range(batch):
            if b not in caches:
                tok_h[b] = int(np.argmax(got[b]))
        pos_h += 1
    return stats
