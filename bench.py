"""Decode benchmark of the persistent megakernel (one JSON line on stdout).

Default workload: the Llama-3-8B-shaped decoder at batch 1 — a 39-token
random prompt followed by greedy decode steps, the single-GPU decode setting
the MPK pages measure (16 GB of weights, 39-token prompt, 512 generated
tokens).  A "step" is one decode step of the whole hot path (embedding,
32 x [RMSNorm+QKV+RoPE, attention with KV append, O+residual,
RMSNorm+gate/up+SiLU*mul, down+residual], final RMSNorm + LM head) plus the
device-side greedy pick of the next token.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mk|reference]

With N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the decode step has no exchange step to shard); the barrier + max over
ranks brackets the timed region.  --impl reference times the fp64 CPU
oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from dataclasses import replace
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import synth  # noqa: E402
from synth import WORKLOADS  # noqa: E402

METRIC = "decode ms/token (batch 1) + achieved HBM GB/s vs B300 peak per step"
FALLBACK_HBM_GBS = 6400.0


def weight_bytes_read(m, batch: int) -> int:
    """bf16 weight bytes one decode step must read: every layer matrix and
    gain, the final gain and the LM head once, one embedding row per sequence."""
    per_layer = sum(int(np.prod(s)) for s in synth.layer_shapes(m).values())
    return 2 * (m.n_layers * per_layer + m.vocab * m.hidden + m.hidden + batch * m.hidden)


def step_bytes(m, batch: int, ctx: int) -> int:
    """Algorithmic HBM bytes of one decode step at context length ctx (the new
    token included): the weights above, every cached K/V entry once, the new
    K/V entry written once, the logits written once."""
    per_tok = 2 * m.n_layers * m.n_kv_heads * m.head_dim * 2  # K and V, all layers, bf16
    return weight_bytes_read(m, batch) + batch * (per_tok * (ctx - 1) + per_tok + m.vocab * 4)


# DRAM bytes (read + write) of one megakernel launch of the full-size
# workload, from ncu captures (dram__bytes_read.sum + dram__bytes_write.sum,
# one pass) of the same workload cut to 2 and 4 layers: the 4-layer launch
# plus 28 times the per-layer difference (the rest of the launch, embedding
# and LM head, is the same at every depth).  Keyed by (workload, batch) and by
# the fingerprint of the kernel sources the captures ran; a source change
# makes the entry stale and the bench line reports null.
NCU_TRAFFIC = {
    ("8b", 1): {"fingerprint": "f85a1c652a69deed", "bytes": 2.818927e9 + 28 * 0.440913e9,
                "summary": "profiles/megakernel_8b_b1_dram.md"},
    ("8b-batch", 64): {"fingerprint": "f85a1c652a69deed", "bytes": 7.195817e9 + 28 * 1.535045e9,
                       "summary": "profiles/megakernel_8b_b64_dram.md"},
}


# the files the megakernel's device code is compiled from (host-side files
# such as the C ABI and the planner do not change its DRAM traffic)
KERNEL_SOURCES = ("megakernel.cu", "mk_kernel.h", "mk_types.h", "ptx.cuh")


def kernel_fingerprint() -> str:
    """sha256 (first 16 hex digits) over the kernel's device sources, file by file."""
    import hashlib
    h = hashlib.sha256()
    root = ROOT / "persistent_decode_megakernel_04_b300" / "csrc"
    for name in KERNEL_SOURCES:
        h.update(name.encode())
        h.update((root / name).read_bytes())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, batch: int, overridden: int):
    """Bytes per launch of the capture above, or None when the workload was
    cut or resized or the kernel sources changed since."""
    e = NCU_TRAFFIC.get((workload, batch))
    if e is None or overridden or e["fingerprint"] != kernel_fingerprint():
        return None
    return e["bytes"]


def measured_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [v for v in (num(r[1]) for r in self.rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in self.rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in self.rows)}


# ----------------------------------------------------------------- CPU side

def _host_budget_bytes() -> int:
    """Host memory the oracle's weights may take: half the machine's RAM."""
    try:
        return os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES") // 2
    except (ValueError, OSError):
        return 32 << 30


def oracle_steps(m, pos0: int, steps: int, warm: int = 1, threads: int = 0, seed: int = 0, model=None):
    """Times WHOLE decode steps of the fp64 oracle, as it stands: every layer
    and the full LM head, at positions pos0, pos0+1, ... (context pos0+1, ...,
    the positions the GPU arm times).  The cache's first pos0 positions hold
    the seeded stand-in contents: a step's cost does not depend on what the
    cache holds, only on its length.  `warm` untimed steps come first; each
    step feeds the previous one's greedy token.  threads > 0 sets the
    oracle's team size.  A model whose weights do not fit half the host's
    memory (the 70B shape) is timed layer by layer, each layer's weights
    generated untimed before its part of the step.
    Returns (list of ms per step, threads used, model)."""
    import oracle

    if threads > 0:
        oracle.set_num_threads(threads)
    streamed = model is None and synth.weight_bytes(m) > _host_budget_bytes()
    if model is None:
        if streamed:
            emb = synth.normal_bf16((m.vocab, m.hidden), seed, synth.TID_EMBED, m.weight_std)
            lm = synth.normal_bf16((m.vocab, m.hidden), seed, synth.TID_LM_HEAD, m.weight_std)
            fin = synth.normal_bf16((m.hidden,), seed, synth.TID_FINAL_NORM, 0.0, 1.0)
            model = oracle.Model(m, {"embed": emb, "lm_head": lm, "final_norm": fin})
        else:
            model = oracle.Model(m, synth.host_weights(m, seed))
    max_seq = pos0 + warm + steps + 1
    if streamed:
        kc = np.zeros((max_seq, m.n_kv_heads, m.head_dim))
        vc = np.zeros_like(kc)
    else:
        kc, vc = model.new_cache(max_seq)
        for l in range(m.n_layers):
            kc[l, :pos0] = synth.bf16_to_f64(synth.host_kv(m, seed, l, "k", 1, pos0)[0])
            vc[l, :pos0] = synth.bf16_to_f64(synth.host_kv(m, seed, l, "v", 1, pos0)[0])
    tok = int(synth.tokens(1, seed, 0, m.vocab)[0])
    times = []
    for i in range(warm + steps):
        if streamed:
            x = model.embed_token(tok)
            dt = 0.0
            for l in range(m.n_layers):
                lw = synth.host_layer_weights(m, seed, l)
                kc[:pos0] = synth.bf16_to_f64(synth.host_kv(m, seed, l, "k", 1, pos0)[0])
                vc[:pos0] = synth.bf16_to_f64(synth.host_kv(m, seed, l, "v", 1, pos0)[0])
                t0 = time.perf_counter()
                model.layer_step(lw, kc, vc, pos0 + i, x)
                dt += time.perf_counter() - t0
            t0 = time.perf_counter()
            logits = model.head(x)
            dt += time.perf_counter() - t0
        else:
            t0 = time.perf_counter()
            logits = model.decode_step(kc, vc, tok, pos0 + i)
            dt = time.perf_counter() - t0
        if i >= warm:
            times.append(dt * 1e3)
        tok = int(np.argmax(logits))
    return times, oracle.num_threads(), model


def cpu_baseline(m, pos0: int, steps: int, single_thread_steps: int):
    """The oracle on all the host cores it runs with by default (`steps`
    whole decode steps) and on one thread (`single_thread_steps` steps), at
    the positions the GPU arm times."""
    import oracle

    default_threads = oracle.num_threads()
    ms, threads, model = oracle_steps(m, pos0, steps)
    out = {"value": statistics.mean(ms), "unit": "ms/token", "cores": threads, "kind": "oracle",
           "sample": f"{steps} whole decode steps of the {m.name} fp64 oracle (every layer, full LM head) at "
                     f"positions {pos0}..{pos0 + steps - 1}, after 1 untimed step"}
    if single_thread_steps > 0:
        ms1, t1, _ = oracle_steps(m, pos0, single_thread_steps, warm=0, threads=1, model=model)
        out["single_thread"] = {"value": statistics.mean(ms1), "unit": "ms/token", "cores": t1,
                                "sample": f"{single_thread_steps} whole decode step(s) from position {pos0}"}
        oracle.set_num_threads(default_threads)
    return out


def run_reference(args, wl):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    m = wl.model
    # the same context lengths as the GPU arm's timed steps: prompt, then the warm-up steps
    pos0 = wl.prompt_len + args.warmup
    ms, threads, _ = oracle_steps(m, pos0, args.steps, warm=args.warmup)
    value = statistics.mean(ms)
    desc = (f"{args.steps} whole decode steps of the {m.name} fp64 oracle (every layer, full LM head) at "
            f"positions {pos0}..{pos0 + args.steps - 1}, after {args.warmup} untimed steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "ms/token", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded random-init weights)",
        "config": {"workload": args.workload, "model": m.name, "batch": wl.batch, "prompt_len": wl.prompt_len,
                   "context": "seeded paged cache" if seeded_context(wl) else "prefilled prompt",
                   "ctx_first_timed": pos0 + 1, "ctx_last_timed": pos0 + args.steps,
                   "parallelism": "replicas x1"},
        "cpu_baseline": {"value": value, "unit": "ms/token", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "ms/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- ranks

class Ranks:
    """One process per GPU under torchrun (RANK, LOCAL_RANK and WORLD_SIZE
    from the environment), or a single process.  Replicas only: no data
    crosses ranks; the timed region is bracketed by barriers and its length
    is the maximum over ranks."""

    def __init__(self, backend: str, device=None):
        import torch.distributed as dist

        self.dist = dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.device = device
        if self.world > 1:
            if backend == "nccl":
                dist.init_process_group(backend, device_id=device)
            else:
                dist.init_process_group(backend)

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, v: float) -> float:
        if self.world == 1:
            return v
        import torch

        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1 and self.dist.is_initialized():
            self.dist.destroy_process_group()


def job_rates(ms_step_max: float, batch: int, world: int):
    """(ms per token of each replica, whole-job tokens/s) from the slowest
    rank's ms per step; every rank decodes `batch` sequences per step."""
    return ms_step_max / batch, 1e3 / ms_step_max * batch * world


# ----------------------------------------------------------------- GPU side

def seeded_context(wl) -> bool:
    """Contexts of 1024 tokens and more are seeded into the paged cache
    instead of prefilled token by token."""
    return wl.prompt_len >= 1024


def time_prefill(mk, plan, m, weights, B, max_seq, prompt_d, kv, logits, reps, popts):
    """Prompt prefill timed with CUDA events: the plan's mk_prefill (the
    chunked-prefill engine below 64 sequences), then the decode step once
    per position (a plan with prefill_by_decode) on the same cache.  Both
    rewrite the same K/V values the first prefill wrote."""
    import torch

    stream = torch.cuda.current_stream()
    T = prompt_d.shape[-1]

    def timed(p):
        p.prefill(prompt_d, kv, logits)  # warm-up (the engine exists already)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            p.prefill(prompt_d, kv, logits)
        b.record(stream)
        torch.cuda.synchronize()
        p.check()
        return a.elapsed_time(b) / reps

    ms = timed(plan)
    kw = {f: getattr(popts, f) for f, _ in popts._fields_ if f != "reserved"} if popts is not None else {}
    ref = mk.Plan(m, weights, batch=B, max_seq=max_seq, opts=mk.mk_plan_options(**{**kw, "prefill_by_decode": 1}))
    ms_dec = timed(ref)
    ref.close()
    return {"tokens": int(T * B), "ms": ms, "tokens_per_s": T * B / ms * 1e3,
            "engine": "chunked (64 tokens per launch)" if B < 64 else "decode step per position",
            "by_decode_ms": ms_dec, "by_decode_tokens_per_s": T * B / ms_dec * 1e3}


def run_mk(args, wl):
    import torch

    import persistent_decode_megakernel_04_b300 as mk

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks("nccl", dev)
    world, rank = ranks.world, ranks.rank
    m = wl.model
    B = wl.batch
    max_seq = ((wl.prompt_len + 2 * args.warmup + args.steps + args.e2e_steps + 4 + 63) // 64) * 64
    weights = synth.device_weights(m, wl.seed, device=dev)
    kw = dict(kv.split("=") for kv in args.plan_opt)
    kw = {k: int(v) for k, v in kw.items()}
    if args.tensor_cores:
        kw["tensor_cores"] = 1
    popts = mk.mk_plan_options(**kw) if kw else None
    plan = mk.Plan(m, weights, batch=B, max_seq=max_seq, opts=popts)
    kv = mk.KVCache(m, B, max_seq, shuffle_seed=1, device=dev)
    logits = torch.empty((B, m.vocab), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    prefill_info = None
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    pos = torch.full((B,), wl.prompt_len - 1, dtype=torch.int32, device=dev)
    if seeded_context(wl):
        # long contexts: the paged cache of positions [0, prompt_len) is filled
        # with seeded values (as if prefilled), then decode starts there
        for l in range(m.n_layers):
            synth.device_kv_pages(kv.k[l], kv.page_table, m, wl.seed, l, "k", B, kv.max_pages, wl.prompt_len,
                                  kv.page_size)
            synth.device_kv_pages(kv.v[l], kv.page_table, m, wl.seed, l, "v", B, kv.max_pages, wl.prompt_len,
                                  kv.page_size)
        tok.copy_(torch.tensor(synth.tokens(B, wl.seed, 0, m.vocab), dtype=torch.int32))
        pos.fill_(wl.prompt_len)
    else:
        prompt = np.stack([synth.tokens(wl.prompt_len, wl.seed, b, m.vocab) for b in range(B)])
        prompt_d = torch.tensor(prompt, dtype=torch.int32, device=dev)
        plan.prefill(prompt_d, kv, logits)
        plan.greedy_next(logits, tok, pos)  # first generated token, at position prompt_len
        if args.prefill_reps > 0:
            prefill_info = time_prefill(mk, plan, m, weights, B, max_seq, prompt_d, kv, logits, args.prefill_reps,
                                        popts)
    for _ in range(args.warmup):
        plan.decode_step(tok, pos, kv, logits)
        plan.greedy_next(logits, tok, pos)
    plan.check()
    ctx0 = wl.prompt_len + args.warmup + 1  # context length (new token included) of the first timed step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The timed steps replay CUDA graphs of the step: a serving loop launches
    # it that way, and for the small shapes the host's per-launch work would
    # otherwise be what is timed.  The greedy pick runs inside the decode
    # launch (mk_decode_step_greedy); --separate-pick times the decode launch
    # and then mk_greedy_next.  Falls back to direct launches if capture is
    # refused.
    fused = not args.separate_pick

    def step_decode():
        if fused:
            plan.decode_step_greedy(tok, pos, kv, logits)
        else:
            plan.decode_step(tok, pos, kv, logits)

    def step_pick():
        if not fused:
            plan.greedy_next(logits, tok, pos)

    launch_mode = "eager"
    g_step = g_pick = None
    if not args.no_graph:
        try:
            g_step, g_pick = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.graph(g_step, stream=cap):
                step_decode()
            if fused:
                g_pick = None
            else:
                with torch.cuda.graph(g_pick, stream=cap):
                    step_pick()
            stream.wait_stream(cap)
            torch.cuda.synchronize()
            plan.check()
            launch_mode = "cuda graph per step"
        except Exception as exc:  # capture refused: time direct launches
            print(f"graph capture unavailable ({exc}); timing direct launches", file=sys.stderr)
            g_step = g_pick = None
            torch.cuda.synchronize()
            plan.check()
    ranks.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            if g_step is not None:
                g_step.replay()
            else:
                step_decode()
            ev[i][1].record(stream)
            if g_pick is not None:
                g_pick.replay()
            else:
                step_pick()
        end.record(stream)
        torch.cuda.synchronize()
    ranks.barrier()
    plan.check()
    ms_step = ranks.max(start.elapsed_time(end) / args.steps)
    kern_ms = [a.elapsed_time(b) for a, b in ev]
    ms_token, tokens_per_s = job_rates(ms_step, B, world)
    bytes_total = sum(step_bytes(m, B, ctx0 + i) for i in range(args.steps))
    achieved = bytes_total / (sum(kern_ms) / 1e3) / 1e9
    peak, peak_src = measured_peak()
    clk = clocks.summary()

    # end to end through the host-buffer entry points, from pinned host
    # memory: (1) the greedy step (tokens and positions in, the picked tokens
    # out; the pick runs in the launch), the `e2e` figure; (2) tokens in,
    # logits out, the argmax on the host, reported beside it
    h_tok = torch.empty(B, dtype=torch.int32).pin_memory()
    h_pos = torch.empty(B, dtype=torch.int32).pin_memory()
    h_nxt = torch.empty(B, dtype=torch.int32).pin_memory()
    h_log = torch.empty((B, m.vocab), dtype=torch.float32).pin_memory()
    h_tok.copy_(tok.cpu())
    h_pos.copy_(pos.cpu())
    n_tok, n_pos, n_nxt, n_log = h_tok.numpy(), h_pos.numpy(), h_nxt.numpy(), h_log.numpy()

    def e2e_greedy():
        plan.decode_step_greedy_host(h_tok, h_pos, kv, h_nxt)
        n_tok[:] = n_nxt
        n_pos[:] += 1

    def e2e_logits():
        plan.decode_step_host(h_tok, h_pos, kv, h_log)
        n_tok[:] = np.argmax(n_log, axis=1)
        n_pos[:] += 1

    def time_e2e(step_fn):
        for _ in range(args.warmup):  # first-call costs stay out of the timed region, as for `value`
            step_fn()
        # the same context lengths as the device-timed steps (their cache slots are rewritten)
        n_pos[:] = ctx0 - 1
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            step_fn()
        return (time.perf_counter() - t0) * 1e3 / args.e2e_steps

    e2e_ms = time_e2e(e2e_greedy)
    e2e_logits_ms = time_e2e(e2e_logits)

    # launch-per-operator ablation of the same task code
    abl = {}
    if args.ablation_steps:
        pos_a, tok_a = h_pos.to(dev), h_tok.to(dev)
        for _ in range(2):
            plan.decode_step_ablation(tok_a, pos_a, kv, logits)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(args.ablation_steps):
            plan.decode_step_ablation(tok_a, pos_a, kv, logits)
        s1.record(stream)
        torch.cuda.synchronize()
        abl["launch_per_op_ms_per_step"] = s0.elapsed_time(s1) / args.ablation_steps
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.decode_step_ablation(tok_a, pos_a, kv, logits)
        g.replay()
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(args.ablation_steps):
            g.replay()
        s1.record(stream)
        torch.cuda.synchronize()
        abl["launch_per_op_graph_ms_per_step"] = s0.elapsed_time(s1) / args.ablation_steps
        abl["launches_per_step"] = 5 * m.n_layers + 1
        abl["ctx"] = int(pos_a[0].item()) + 1
        plan.check()

    if args.trace_out and rank == 0:
        # one more step with a tracing plan over the same weights and cache
        from persistent_decode_megakernel_04_b300 import trace as mktrace

        topt = mk.mk_plan_options(**{**kw, "trace": 1})
        tplan = mk.Plan(m, weights, batch=B, max_seq=max_seq, opts=topt)
        tpos = h_pos.to(dev)
        for _ in range(2):
            tplan.decode_step(h_tok.to(dev), tpos, kv, logits)
        tr = tplan.trace()
        tplan.check()
        tasks, _ = mk.mk_plan_describe(tplan.cfg, tr.shape[0], topt)
        rows = mktrace.phases(tasks, tr)
        Path(args.trace_out).write_text(json.dumps(rows, indent=1))
        Path(args.trace_out).with_suffix(".chrome.json").write_text(mktrace.chrome_trace(tasks, tr))
        np.save(Path(args.trace_out).with_suffix(".raw.npy"), tr)  # [cta][queue position][8] stamps
        tplan.close()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(m, ctx0 - 1, args.cpu_samples, args.cpu_single_thread_steps)

    if rank == 0:
        line = {
            "metric": METRIC, "value": ms_token, "unit": "ms/token", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 weights/KV, fp32 math",
            "data": "synthetic (seeded random-init weights, random prompt ids)",
            "config": {"workload": args.workload, "model": m.name, "batch": B, "prompt_len": wl.prompt_len,
                       "context": "seeded paged cache" if seeded_context(wl) else "prefilled prompt",
                       "projections": "tcgen05 tiles" if (B > 1 or args.tensor_cores) else "CUDA-core matvec",
                       "ctx_first_timed": ctx0, "ctx_last_timed": ctx0 + args.steps - 1,
                       "parallelism": f"replicas x{world}", "launch": launch_mode,
                       "greedy_pick": "in the decode launch" if fused else "separate kernel",
                       **({"plan_options": kw} if kw else {}),
                       "l2": f"no flush: {weight_bytes_read(m, B) / 1e9:.1f} GB of weights stream per step (> 126 MB L2)"},
            "tokens_per_s": tokens_per_s,
            "hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": ncu_traffic(args.workload, B, args.layers or args.prompt_len),
                         "kernel": "megakernel", "kernel_ms_mean": statistics.mean(kern_ms),
                         "bytes_per_step_mean": bytes_total / args.steps},
            "clocks": clk,
            "e2e": {"value": e2e_ms / B, "unit": "ms/token", "h2d_bytes_per_step": 8 * B,
                    "d2h_bytes_per_step": 4 * B, "api": "mk_decode_step_greedy_host",
                    "logits_to_host": {"value": e2e_logits_ms / B, "unit": "ms/token", "h2d_bytes_per_step": 8 * B,
                                       "d2h_bytes_per_step": 4 * B * m.vocab,
                                       "api": "mk_decode_step_host + host argmax"}},
            "gpu_launches": (1 if fused else 2) * args.steps,
            "ablation": abl,
            "prefill": prefill_info,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    plan.close()
    ranks.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mk", "reference"], default="mk")
    ap.add_argument("--workload", default="8b", choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=32)
    ap.add_argument("--ablation-steps", type=int, default=8)
    ap.add_argument("--cpu-samples", type=int, default=8, help="whole oracle decode steps timed on all host cores")
    ap.add_argument("--prefill-reps", type=int, default=3, help="prompt prefills timed (0: skip)")
    ap.add_argument("--cpu-single-thread-steps", type=int, default=1,
                    help="whole oracle decode steps timed on one host thread (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prompt-len", type=int, default=0, help="override the workload's prompt length")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (sequences per step)")
    ap.add_argument("--layers", type=int, default=0, help="profiling only: keep the shape, use this many layers")
    ap.add_argument("--tensor-cores", action="store_true",
                    help="run the projections as tcgen05 tiles at batch 1 too (default: CUDA-core matvecs)")
    ap.add_argument("--no-graph", action="store_true", help="time direct launches instead of CUDA graph replays")
    ap.add_argument("--separate-pick", action="store_true",
                    help="time the decode launch and mk_greedy_next instead of the pick fused into the decode launch")
    ap.add_argument("--plan-opt", action="append", default=[], metavar="FIELD=INT",
                    help="set an mk_plan_options field (tuning sweeps), e.g. max_inflight=3")
    ap.add_argument("--trace-out", default="", help="write a per-phase task trace of one extra step here")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = WORKLOADS[args.workload]
    if args.prompt_len > 0:
        wl = replace(wl, prompt_len=args.prompt_len)
    if args.batch > 0:
        wl = replace(wl, batch=args.batch)
    if args.layers > 0:
        # profiling a full-width model with fewer layers (the measured workload keeps every layer)
        wl = replace(wl, model=replace(wl.model, n_layers=args.layers, name=f"{wl.model.name}-{args.layers}l"))
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_mk(args, wl)


if __name__ == "__main__":
    main()
