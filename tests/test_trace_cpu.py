"""Per-phase summaries and Chrome-trace JSON of a task trace, on the CPU:
a real task graph (mk_plan_describe, no GPU) with synthetic stamps whose
phase boundaries, waits and skipped tasks are known."""
from __future__ import annotations

import json
from collections import defaultdict

import numpy as np

import persistent_decode_megakernel_04_b300 as mk
from persistent_decode_megakernel_04_b300 import trace as mktrace
from synth import WORKLOADS

NUM_CTAS = 6
T0 = 1_000_000_000  # globaltimer nanoseconds of the step's first start


def _graph():
    m = WORKLOADS["tiny"].model
    tasks, _ = mk.mk_plan_describe(mk.model_cfg(m, 1, 256), NUM_CTAS, None)
    return m, tasks


def _stamps(tasks, skip=()):
    """Task number k (global queue order) of stage s = (layer, op) starts at
    T0 + 10 us * s_index + 100 ns * k, runs 2 us, was released 500 ns before
    it started, waited 300 ns for data and 700 ns for a free slot."""
    stages = sorted({(t.layer, t.op) for t in tasks}, key=lambda s: (s[0], s[1] == mk.OP_LM, s[1]))
    order = {s: i for i, s in enumerate(stages)}
    by_cta = defaultdict(list)
    for t in tasks:
        by_cta[t.cta].append(t)
    max_tasks = max(len(q) for q in by_cta.values())
    tr = np.zeros((NUM_CTAS, max_tasks, 8), dtype=np.uint64)
    k = 0
    expect = {}
    for cta in range(NUM_CTAS):
        for i, t in enumerate(by_cta[cta]):
            k += 1
            if (cta, i) in skip:
                continue
            start = T0 + 10_000 * order[(t.layer, t.op)] + 100 * k
            tr[cta, i] = [start - 500, start, start + 2_000, 300, 0, 700, 0, 0]
            expect.setdefault((t.layer, t.op), []).append(start)
    return tr, expect


def test_phase_rows_match_the_stamps():
    m, tasks = _graph()
    tr, expect = _stamps(tasks)
    rows = mktrace.phases(tasks, tr)
    assert len(rows) == len(expect)
    t0 = min(min(v) for v in expect.values())
    names = {v: k for k, v in mktrace.OP_NAMES.items()}
    for r in rows:
        starts = expect[(r["layer"], names[r["op"]])]
        assert r["tasks"] == len(starts)
        assert r["first_start_us"] == (min(starts) - t0) / 1e3
        assert r["last_end_us"] == (max(starts) + 2_000 - t0) / 1e3
        assert r["first_release_us"] == (min(starts) - 500 - t0) / 1e3
        assert abs(r["mean_task_us"] - 2.0) < 1e-12 and abs(r["max_task_us"] - 2.0) < 1e-12
        assert abs(r["mean_data_wait_us"] - 0.3) < 1e-12 and abs(r["mean_ring_full_us"] - 0.7) < 1e-12
    # rows come out in order of their first start: layer by layer, operator by operator
    firsts = [r["first_start_us"] for r in rows]
    assert firsts == sorted(firsts)
    assert rows[0]["op"] == "qkv" and rows[-1]["op"] == "lm_head"


def test_tasks_not_run_are_left_out():
    m, tasks = _graph()
    skip = {(0, 0), (1, 2)}
    tr, expect = _stamps(tasks, skip=skip)
    rows = mktrace.phases(tasks, tr)
    assert sum(r["tasks"] for r in rows) == len(tasks) - len(skip)
    ev = json.loads(mktrace.chrome_trace(tasks, tr))["traceEvents"]
    assert len(ev) == len(tasks) - len(skip)


def test_chrome_trace_events():
    m, tasks = _graph()
    tr, expect = _stamps(tasks)
    doc = json.loads(mktrace.chrome_trace(tasks, tr))
    ev = doc["traceEvents"]
    assert len(ev) == len(tasks)
    assert {e["tid"] for e in ev} == {t.cta for t in tasks}
    assert min(e["ts"] for e in ev) == 0.0
    assert all(e["ph"] == "X" and abs(e["dur"] - 2.0) < 1e-12 for e in ev)
    attn = [e for e in ev if e["name"].endswith(" attn")]
    assert attn and all({"seq", "kv_head", "split"} <= set(e["args"]) for e in attn)
    proj = [e for e in ev if not e["name"].endswith(" attn")]
    assert all(e["args"]["rows"][0] < e["args"]["rows"][1] for e in proj)
