"""Task traces of the megakernel: per-phase summaries and Chrome-trace JSON.

A plan created with ``mk_plan_options(trace=1)`` stamps every task with the
global timer (see ``mk_plan_trace`` in include/mk.h).  The queue order of the
stamps is the order ``mk_plan_describe`` returns for the same options, which
is how each stamp is matched to its (layer, operator, rows) here.
"""
from __future__ import annotations

import json
from collections import defaultdict

import numpy as np

OP_NAMES = {1: "qkv", 2: "attn", 3: "o", 4: "gate_up", 5: "down", 6: "lm_head", 7: "embed", 8: "kv_append"}


def _by_cta(tasks):
    q = defaultdict(list)
    for t in tasks:
        q[t.cta].append(t)
    return q


def phases(tasks, trace: np.ndarray) -> list:
    """One row per (layer, op): first release, last release, first start,
    last end, mean compute-side data wait and mean producer ring-full wait,
    all in microseconds relative to the earliest stamp of the step."""
    t0 = int(trace[..., 1][trace[..., 1] > 0].min())
    acc = defaultdict(lambda: {"rel": [], "start": [], "end": [], "wait": [], "ring_full": [], "dur": [],
                               "act_wait": [], "acc_wait": []})
    for cta, q in _by_cta(tasks).items():
        for i, t in enumerate(q):
            e = trace[cta, i]
            if e[2] == 0:
                continue
            a = acc[(t.layer, t.op)]
            a["rel"].append((int(e[0]) - t0) / 1e3 if e[0] else None)
            a["start"].append((int(e[1]) - t0) / 1e3)
            a["end"].append((int(e[2]) - t0) / 1e3)
            a["dur"].append((int(e[2]) - int(e[1])) / 1e3)
            a["wait"].append(int(e[3]) / 1e3)
            a["ring_full"].append(int(e[5]) / 1e3)
            a["act_wait"].append(int(e[6]) / 1e3)
            a["acc_wait"].append(int(e[7]) / 1e3)
    rows = []
    for (layer, op), a in sorted(acc.items(), key=lambda kv: min(kv[1]["start"])):
        rel = [r for r in a["rel"] if r is not None]
        rows.append({
            "layer": layer, "op": OP_NAMES.get(op, str(op)), "tasks": len(a["start"]),
            "first_release_us": min(rel) if rel else None, "last_release_us": max(rel) if rel else None,
            "first_start_us": min(a["start"]), "last_end_us": max(a["end"]),
            "mean_task_us": float(np.mean(a["dur"])), "max_task_us": float(np.max(a["dur"])),
            "mean_data_wait_us": float(np.mean(a["wait"])), "mean_ring_full_us": float(np.mean(a["ring_full"])),
            "mean_act_wait_us": float(np.mean(a["act_wait"])), "mean_acc_wait_us": float(np.mean(a["acc_wait"])),
        })
    return rows


def chrome_trace(tasks, trace: np.ndarray) -> str:
    """Chrome-trace (about://tracing, Perfetto) JSON: one row per worker CTA."""
    t0 = int(trace[..., 1][trace[..., 1] > 0].min())
    ev = []
    for cta, q in _by_cta(tasks).items():
        for i, t in enumerate(q):
            e = trace[cta, i]
            if e[2] == 0:
                continue
            name = f"L{t.layer} {OP_NAMES.get(t.op, t.op)}"
            args = {"rows": [t.a0, t.a1], "data_wait_us": int(e[3]) / 1e3, "ring_full_us": int(e[5]) / 1e3}
            if t.op == 2:
                args = {"seq": t.a0, "kv_head": t.a1, "split": t.a2, "data_wait_us": int(e[3]) / 1e3}
            ev.append({"name": name, "ph": "X", "pid": 0, "tid": cta, "ts": (int(e[1]) - t0) / 1e3,
                       "dur": (int(e[2]) - int(e[1])) / 1e3, "args": args})
    return json.dumps({"traceEvents": ev, "displayTimeUnit": "ns"})
