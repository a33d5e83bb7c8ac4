"""Host task-graph builder: coverage, event thresholds and a simulated run of
the per-CTA queues (the device runtime's semantics, executed on the CPU)."""
from collections import defaultdict

import pytest

import persistent_decode_megakernel_04_b300 as mk
from synth import WORKLOADS

SHAPES = {
    "tiny": WORKLOADS["tiny"].model,
    "1b": WORKLOADS["1b"].model,
    "8b": WORKLOADS["8b"].model,
}


def describe(name, num_ctas, **kw):
    m = SHAPES[name]
    cfg = mk.model_cfg(m, 1, 1024)
    opts = mk.mk_plan_options(**kw) if kw else None
    tasks, n_events = mk.mk_plan_describe(cfg, num_ctas, opts)
    return m, tasks, n_events


def op_rows(m, op):
    d = m.head_dim
    return {mk.OP_QKV: (m.n_q_heads + 2 * m.n_kv_heads) * d, mk.OP_O: m.hidden, mk.OP_GU: m.ffn_dim,
            mk.OP_DOWN: m.hidden, mk.OP_LM: m.vocab}[op]


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("num_ctas", [148, 37, 1])
def test_every_output_row_covered_exactly_once(name, num_ctas):
    m, tasks, _ = describe(name, num_ctas)
    cover = defaultdict(list)
    for t in tasks:
        if t.op != mk.OP_ATTN:
            cover[(t.layer, t.op)].append((t.a0, t.a1))
    for l in range(m.n_layers):
        for op in (mk.OP_QKV, mk.OP_O, mk.OP_GU, mk.OP_DOWN):
            rs = sorted(cover[(l, op)])
            assert rs[0][0] == 0 and rs[-1][1] == op_rows(m, op)
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:])), "gap or overlap"
            sizes = [b - a for a, b in rs]
            assert max(sizes) - min(sizes) <= 1, "row ranges balanced to one row"
    lm = sorted(cover[(m.n_layers - 1, mk.OP_LM)])
    assert lm[0][0] == 0 and lm[-1][1] == m.vocab


@pytest.mark.parametrize("name", list(SHAPES))
def test_attention_tasks_cover_every_head_and_split(name):
    m, tasks, _ = describe(name, 148)
    att = [t for t in tasks if t.op == mk.OP_ATTN]
    S = att[0].a3
    assert S == min(64, max(1, 148 // m.n_kv_heads))  # default splits, capped at 64
    seen = {(t.layer, t.a0, t.a1, t.a2) for t in att}
    assert len(seen) == len(att) == m.n_layers * m.n_kv_heads * S


def test_queue_order_is_stage_order_within_each_cta():
    _, tasks, _ = describe("8b", 148)
    stage = lambda t: (t.layer, t.op)
    by_cta = defaultdict(list)
    for t in tasks:
        by_cta[t.cta].append(stage(t))
    for q in by_cta.values():
        assert q == sorted(q)


def simulate(m, tasks, n_events):
    """Runs the queues with event counters as the device does: a CTA's next task
    may run once counter[wait] >= wait_count; attention signals once per
    (sequence, kv head), when its last split finishes."""
    queues = defaultdict(list)
    for t in tasks:
        queues[t.cta].append(t)
    head = {c: 0 for c in queues}
    ctr = [0] * n_events
    done_splits = defaultdict(int)
    order = []
    progress = True
    while progress:
        progress = False
        for c, q in queues.items():
            while head[c] < len(q):
                t = q[head[c]]
                if t.wait_event >= 0 and ctr[t.wait_event] < t.wait_count:
                    break
                if t.op == mk.OP_ATTN:
                    k = (t.layer, t.a0, t.a1)
                    done_splits[k] += 1
                    if done_splits[k] == t.a3:
                        ctr[t.signal_event] += 1
                elif t.signal_event >= 0:
                    ctr[t.signal_event] += 1
                order.append(t)
                head[c] += 1
                progress = True
    return all(head[c] == len(q) for c, q in queues.items()), order, ctr


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("num_ctas,seed", [(148, 0), (148, 7), (5, 3)])
def test_schedule_completes_and_respects_dependencies(name, num_ctas, seed):
    m, tasks, n_events = describe(name, num_ctas, planner_seed=seed)
    ok, order, ctr = simulate(m, tasks, n_events)
    assert ok, "deadlock: some queue never drained"
    expect = {}
    for t in tasks:
        if t.wait_event >= 0:
            assert expect.setdefault(t.wait_event, t.wait_count) == t.wait_count
    for e, cnt in expect.items():
        assert ctr[e] == cnt
    pos = {}
    for i, t in enumerate(order):
        pos.setdefault((t.layer, t.op), []).append(i)
    for l in range(m.n_layers):
        assert min(pos[(l, mk.OP_ATTN)]) > max(pos[(l, mk.OP_QKV)])
        assert min(pos[(l, mk.OP_O)]) > max(pos[(l, mk.OP_ATTN)])
        assert min(pos[(l, mk.OP_GU)]) > max(pos[(l, mk.OP_O)])
        assert min(pos[(l, mk.OP_DOWN)]) > max(pos[(l, mk.OP_GU)])
        if l + 1 < m.n_layers:
            assert min(pos[(l + 1, mk.OP_QKV)]) > max(pos[(l, mk.OP_DOWN)])


def test_unreachable_event_option_blocks_the_schedule():
    m, tasks, n_events = describe("tiny", 148, test_unreachable_event=2)
    ok, _, _ = simulate(m, tasks, n_events)
    assert not ok


def test_planner_seed_permutes_assignment_but_not_work():
    _, a, _ = describe("tiny", 148)
    _, b, _ = describe("tiny", 148, planner_seed=11)
    key = lambda t: (t.layer, t.op, t.a0, t.a1, t.a2)
    assert sorted(map(key, a)) == sorted(map(key, b))
    assert [t.cta for t in sorted(a, key=key)] != [t.cta for t in sorted(b, key=key)]


# ------------------------------------------------------------ batched path

def describe_b(name, B, num_ctas, **kw):
    m = SHAPES[name]
    cfg = mk.model_cfg(m, B, 1024)
    opts = mk.mk_plan_options(**kw) if kw else None
    tasks, n_events = mk.mk_plan_describe(cfg, num_ctas, opts)
    return m, tasks, n_events


def tc_sub_default(B):
    """64-column K sub-tiles per projection unit by default."""
    return 2


def tc_units(m, op, B=64):
    T, K = mk.TC_TILE_M, mk.TC_TILE_K * tc_sub_default(B)
    cdiv = lambda a, b: (a + b - 1) // b
    d = m.head_dim
    if op == mk.OP_QKV:
        tiles = cdiv(m.n_q_heads * d, T) + 2 * cdiv(m.n_kv_heads * d, T)
        return tiles * cdiv(m.hidden, K), cdiv(m.hidden, K)
    rows, k = {mk.OP_O: (m.hidden, m.n_q_heads * d), mk.OP_GU: (m.ffn_dim, m.hidden),
               mk.OP_DOWN: (m.hidden, m.ffn_dim), mk.OP_LM: (m.vocab, m.hidden)}[op]
    return cdiv(rows, T) * cdiv(k, K), cdiv(k, K)


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("B,num_ctas", [(2, 148), (64, 148), (16, 37), (8, 1)])
def test_batched_units_covered_once_and_balanced(name, B, num_ctas):
    m, tasks, _ = describe_b(name, B, num_ctas)
    cover = defaultdict(list)
    for t in tasks:
        if t.op not in (mk.OP_ATTN,):
            cover[(t.layer, t.op)].append((t.a0, t.a1, t.a2))
    for l in range(m.n_layers):
        for op in (mk.OP_QKV, mk.OP_O, mk.OP_GU, mk.OP_DOWN):
            U, _ = tc_units(m, op, B)
            rs = sorted(cover[(l, op)])
            assert rs[0][0] == 0 and rs[-1][1] == U
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:])), "gap or overlap"
            sizes = [b - a for a, b, _ in rs]
            assert max(sizes) - min(sizes) <= 1
            # range number c owns [c*U/N, (c+1)*U/N)
            for a0, a1, c in rs:
                assert (a0, a1) == (c * U // num_ctas, (c + 1) * U // num_ctas)
    emb = sorted(cover[(0, mk.OP_EMBED)])
    h_tiles = (m.hidden + mk.TC_TILE_M - 1) // mk.TC_TILE_M
    assert emb[0][0] == 0 and emb[-1][1] == B * h_tiles


@pytest.mark.parametrize("U,N", [(16, 148), (3072, 148), (64128, 148), (7168, 37), (100, 7), (5, 5)])
def test_stream_k_tile_contributors(U, N):
    """The device finds the ranges sharing a row tile from closed forms:
    range_of(u) = ((u+1)N - 1) div U owns unit u, range_start(c) = cU div N.
    Checked against the ranges themselves."""
    starts = [c * U // N for c in range(N + 1)]
    owner = {}
    for c in range(N):
        for u in range(starts[c], starts[c + 1]):
            owner[u] = c
    for u in range(U):
        assert ((u + 1) * N - 1) // U == owner[u]


@pytest.mark.parametrize("name", ["tiny", "8b"])
@pytest.mark.parametrize("B,num_ctas,seed", [(8, 148, 0), (64, 148, 3), (4, 5, 1)])
def test_batched_schedule_completes(name, B, num_ctas, seed):
    m, tasks, n_events = describe_b(name, B, num_ctas, planner_seed=seed)
    assert n_events == 5 * m.n_layers + 1
    ok, order, _ = simulate(m, tasks, n_events)
    assert ok, "deadlock: some queue never drained"
    pos = {}
    for i, t in enumerate(order):
        pos.setdefault((t.layer, t.op), []).append(i)
    assert min(pos[(0, mk.OP_QKV)]) > max(pos[(0, mk.OP_EMBED)])
    for l in range(m.n_layers):
        assert min(pos[(l, mk.OP_ATTN)]) > max(pos[(l, mk.OP_QKV)])
        assert min(pos[(l, mk.OP_DOWN)]) > max(pos[(l, mk.OP_GU)])


@pytest.mark.parametrize("S", [1, 3, 18, 64])
@pytest.mark.parametrize("pos", [0, 1, 63, 64, 65, 130, 4096, 4159])
def test_attention_splits_cover_cached_blocks_once(S, pos):
    """Attention reads the cached context [0, pos) in aligned 64-token blocks;
    split s of S takes blocks [s*nb/S, (s+1)*nb/S) (the device's arithmetic),
    so every cached token is read by exactly one split, and the last split
    alone attends to the new token at pos."""
    nb = (pos + 63) // 64
    seen = []
    for s in range(S):
        seen += list(range(s * nb // S, (s + 1) * nb // S))
    assert seen == list(range(nb))
    covered = {t for b in seen for t in range(64 * b, 64 * b + 64) if t < pos}
    assert covered == set(range(pos))


@pytest.mark.parametrize("batch", [1, 64])
def test_kv_append_graph_orders_append_between_qkv_and_attention(batch):
    """The kv-append graph (the chunked-prefill engine's): per layer one
    append item per (row, kv head), after every QKV task and before every
    attention task, with the schedule still draining."""
    m = SHAPES["8b"]
    cfg = mk.model_cfg(m, batch, 1024)
    tasks, n_events = mk.mk_plan_describe(cfg, 148, mk.mk_plan_options(kv_append=1, tensor_cores=1))
    kva = [t for t in tasks if t.op == mk.OP_KVA]
    for l in range(m.n_layers):
        items = sorted((t.a0, t.a1) for t in kva if t.layer == l)
        assert items[0][0] == 0 and items[-1][1] == batch * m.n_kv_heads
        assert all(a[1] == b[0] for a, b in zip(items, items[1:]))
    ok, order, _ = simulate(m, tasks, n_events)
    assert ok, "deadlock"
    pos = defaultdict(list)
    for i, t in enumerate(order):
        pos[(t.layer, t.op)].append(i)
    for l in range(m.n_layers):
        assert min(pos[(l, mk.OP_KVA)]) > max(pos[(l, mk.OP_QKV)])
        assert min(pos[(l, mk.OP_ATTN)]) > max(pos[(l, mk.OP_KVA)])
    att = [t for t in tasks if t.op == mk.OP_ATTN]
    kva_ev = {t.signal_event for t in kva}
    assert all(t.wait_event in kva_ev for t in att)


def simulate_jit(tasks, n_events, n_ctas, seed, ring=8):
    """Dynamic dispatch as the device runs it: each CTA claims the next
    unclaimed task of the earliest stage with any left (at most `ring`
    claimed and not yet released: a ring slot is reused only once its task
    is released and taken), and runs its claims in claim order once each
    one's event reaches its threshold; CTAs act in a random order."""
    import random

    rnd = random.Random(seed)
    stages, cur = [], None
    for t in tasks:  # stage = a run of tasks of one (layer, op)
        if (t.layer, t.op) != cur:
            stages.append([])
            cur = (t.layer, t.op)
        stages[-1].append(t)
    nxt = [0] * len(stages)
    stage = 0
    claimed = defaultdict(list)
    ctr = [0] * n_events
    done_splits = defaultdict(int)
    order, ran = [], 0
    while ran < len(tasks):
        progress = False
        for c in rnd.sample(range(n_ctas), n_ctas):
            if len(claimed[c]) < ring and stage < len(stages) and rnd.random() < 0.7:
                while stage < len(stages) and nxt[stage] >= len(stages[stage]):
                    stage += 1
                if stage < len(stages):
                    claimed[c].append(stages[stage][nxt[stage]])
                    nxt[stage] += 1
                    progress = True
            if claimed[c]:
                t = claimed[c][0]
                if t.wait_event < 0 or ctr[t.wait_event] >= t.wait_count:
                    claimed[c].pop(0)
                    if t.op == mk.OP_ATTN:
                        k = (t.layer, t.a0, t.a1)
                        done_splits[k] += 1
                        if done_splits[k] == t.a3:
                            ctr[t.signal_event] += 1
                    elif t.signal_event >= 0:
                        ctr[t.signal_event] += 1
                    order.append(t)
                    ran += 1
                    progress = True
        if not progress:
            return False, order
    return True, order


@pytest.mark.parametrize("jit,num_ctas,seed", [(1, 148, 0), (2, 148, 1), (4, 37, 2), (1, 5, 3)])
def test_dynamic_dispatch_graph_completes_under_any_claim_order(jit, num_ctas, seed):
    """Dynamic dispatch (options.jit): no task is bound to a CTA, stages are
    contiguous in stage order, projections are cut into jit ranges per CTA,
    and a randomised run of the claim-and-run rule drains every task with
    the dependencies respected."""
    m = SHAPES["8b"]
    cfg = mk.model_cfg(m, 1, 1024)
    tasks, n_events = mk.mk_plan_describe(cfg, num_ctas, mk.mk_plan_options(jit=jit))
    assert all(t.cta == -1 for t in tasks)
    qkv = [t for t in tasks if t.op == mk.OP_QKV and t.layer == 0]
    rows = op_rows(m, mk.OP_QKV)
    assert len(qkv) == min(rows, jit * num_ctas)
    ok, order = simulate_jit(tasks, n_events, num_ctas, seed)
    assert ok, "deadlock"
    pos = defaultdict(list)
    for i, t in enumerate(order):
        pos[(t.layer, t.op)].append(i)
    for l in range(m.n_layers):
        assert min(pos[(l, mk.OP_ATTN)]) > max(pos[(l, mk.OP_QKV)])
        assert min(pos[(l, mk.OP_O)]) > max(pos[(l, mk.OP_ATTN)])
        assert min(pos[(l, mk.OP_GU)]) > max(pos[(l, mk.OP_O)])
        assert min(pos[(l, mk.OP_DOWN)]) > max(pos[(l, mk.OP_GU)])


def test_dynamic_dispatch_rejects_tracing():
    cfg = mk.model_cfg(SHAPES["tiny"], 1, 128)
    with pytest.raises(mk.MKError):
        mk.mk_plan_describe(cfg, 148, mk.mk_plan_options(jit=1, trace=1))


@pytest.mark.parametrize("split", [1, 2, 3])
def test_tile_split_bounds_the_ranges_per_row_tile(split):
    """tc_tile_split: a tensor-core projection is cut into at most
    tiles * split ranges (all CTAs when that is more), each 128-row tile is
    shared by at most split ranges, the ranges tile the units exactly, a
    stage of fewer ranges than CTAs starts on the CTA after the previous
    stage's last, and the schedule still drains."""
    m = SHAPES["8b"]
    N, B = 148, 64
    cfg = mk.model_cfg(m, B, 4160)
    tasks, n_events = mk.mk_plan_describe(cfg, N, mk.mk_plan_options(tc_tile_split=split))
    H, I, V, d = m.hidden, m.ffn_dim, m.vocab, m.head_dim
    qkv_tiles = (m.n_q_heads * d + 127) // 128 + 2 * ((m.n_kv_heads * d + 127) // 128)
    kw = 64 * tc_sub_default(B)  # K columns per unit
    geo = {mk.OP_QKV: (qkv_tiles, H // kw), mk.OP_O: (H // 128, m.n_q_heads * d // kw),
           mk.OP_GU: (I // 128, H // kw), mk.OP_DOWN: (H // 128, I // kw), mk.OP_LM: ((V + 127) // 128, H // kw)}
    for op, (tiles, kchunks) in geo.items():
        ts = sorted((t for t in tasks if t.op == op and t.layer == (m.n_layers - 1 if op == mk.OP_LM else 3)),
                    key=lambda t: t.a0)
        assert len(ts) == min(N, tiles * split), (op, len(ts))
        assert ts[0].a0 == 0 and ts[-1].a1 == tiles * kchunks
        assert all(a.a1 == b.a0 for a, b in zip(ts, ts[1:]))
        assert sorted(t.a2 for t in ts) == list(range(len(ts)))  # range numbers
        assert len({t.cta for t in ts}) == len(ts)  # one range per CTA
        for tile in range(tiles):
            lo, hi = tile * kchunks, (tile + 1) * kchunks
            assert sum(1 for t in ts if t.a0 < hi and t.a1 > lo) <= max(split, -(-len(ts) // tiles) + 1)
    # the O projection of a layer starts on the CTA after the attention tasks' last
    n_att = sum(1 for t in tasks if t.op == mk.OP_ATTN and t.layer == 3)
    o = [t for t in tasks if t.op == mk.OP_O and t.layer == 3]
    if len(o) < N:
        assert min(o, key=lambda t: t.a2).cta == n_att % N
    ok, _, _ = simulate(m, tasks, n_events)
    assert ok, "deadlock"


@pytest.mark.parametrize("B,sub", [(8, 1), (8, 2), (64, 1), (64, 2)])
def test_k_subtiles_set_the_unit_width(B, sub):
    """tc_k_subtiles: a projection unit spans sub 64-column K sub-tiles, so
    each operator has tiles * ceil(K / (64 sub)) units, covered once."""
    m = SHAPES["8b"]
    cfg = mk.model_cfg(m, B, 1024)
    tasks, _ = mk.mk_plan_describe(cfg, 148, mk.mk_plan_options(tc_k_subtiles=sub))
    cdiv = lambda a, b: (a + b - 1) // b
    for op, (rows, K) in {mk.OP_O: (m.hidden, m.n_q_heads * m.head_dim), mk.OP_DOWN: (m.hidden, m.ffn_dim),
                          mk.OP_GU: (m.ffn_dim, m.hidden)}.items():
        rs = sorted((t.a0, t.a1) for t in tasks if t.op == op and t.layer == 0)
        assert rs[0][0] == 0 and rs[-1][1] == cdiv(rows, 128) * cdiv(K, 64 * sub)
        assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))


@pytest.mark.parametrize("B,N", [(64, 148), (32, 148), (16, 37), (20, 148)])
def test_leftover_attention_pairs_are_split_to_even_the_ctas(B, N):
    """With more (sequence, kv head) pairs than CTAs and the default single
    split, the pairs left over after whole rounds are cut into k splits: every
    pair is covered by its splits exactly once, and no CTA carries more than
    the even share rounded up to 1/k of a pair (a whole extra pair before)."""
    m = SHAPES["8b"]
    cfg = mk.model_cfg(m, B, 4160)
    tasks, n_events = mk.mk_plan_describe(cfg, N, mk.mk_plan_options(num_ctas=N))
    att = [t for t in tasks if t.op == mk.OP_ATTN and t.layer == 0]
    P = B * m.n_kv_heads
    pairs = defaultdict(list)
    for t in att:
        pairs[(t.a0, t.a1)].append((t.a2, t.a3))
    assert len(pairs) == P
    for sp in pairs.values():
        k = sp[0][1]
        assert sorted(s for s, _ in sp) == list(range(k)) and all(kk == k for _, kk in sp)
    load = defaultdict(float)
    for t in att:
        load[t.cta] += 1.0 / t.a3
    R = P % N
    ks = {sp[0][1] for sp in pairs.values()}
    if P > N and R:
        k = max(ks)
        assert ks <= {1, k} and k <= 8
        assert max(load.values()) <= P // N + (-(-R * k // N)) / k + 1e-9
    if (B, N) == (64, 148):
        assert ks == {1, 2} and max(load.values()) == 3.5  # 444 whole pairs, 68 in halves
    ok, _, _ = simulate(m, tasks, n_events)
    assert ok, "deadlock"
