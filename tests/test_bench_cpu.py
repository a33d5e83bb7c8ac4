"""The bench's reference arm (the fp64 oracle timed on host cores) and its
JSON line, on the CPU: the line carries the fields every bench line carries,
and ranks other than 0 print nothing and exit 0."""
from __future__ import annotations

import json
import os
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]


def _run(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--workload", "tiny",
                           "--steps", "4", "--warmup", "3", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run()
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "ms/token" and d["higher_is_better"] is False
    assert d["value"] > 0 and d["ms_per_step"] == d["value"]
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny" and d["config"]["ctx_last_timed"] - d["config"]["ctx_first_timed"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "ms/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_no_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def _free_port() -> int:
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica_rank(rank: int, world: int, port: int, out_dir: str):
    """One bench rank on the CPU (gloo): barriers around a 'timed region' whose
    length differs per rank, then the maximum over ranks."""
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, str(ROOT))
    import bench

    ranks = bench.Ranks("gloo")
    assert (ranks.world, ranks.rank) == (world, rank)
    ranks.barrier()
    ms_step = 3.0 + rank  # rank r "took" 3 + r ms per step
    ms_max = ranks.max(ms_step)
    ranks.barrier()
    ms_token, tok_s = bench.job_rates(ms_max, 4, world)
    Path(out_dir, f"rank{rank}.json").write_text(json.dumps([ms_max, ms_token, tok_s]))
    ranks.close()


def test_two_replica_ranks_take_the_slowest_rank_on_gloo(tmp_path):
    import torch.multiprocessing as tmp

    world = 2
    tmp.spawn(_replica_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(world)]
    for ms_max, ms_token, tok_s in got:
        assert ms_max == 4.0  # the slower rank's time, seen by every rank
        assert ms_token == 1.0  # 4 sequences per step on each replica
        assert abs(tok_s - 1e3 / 4.0 * 4 * world) < 1e-9  # both replicas' tokens


def test_single_process_ranks_need_no_process_group():
    sys.path.insert(0, str(ROOT))
    import bench

    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        r = bench.Ranks("gloo")
        assert (r.world, r.rank) == (1, 0)
        r.barrier()
        assert r.max(2.5) == 2.5
        r.close()
    finally:
        os.environ.update(env)


def _hand_weight_bytes(L, H, nq, nkv, d, I, V, batch):
    """bf16 bytes of one step's weights, written out from the decoder's
    matrices: Wq, Wo (nq*d x H), Wk, Wv (nkv*d x H), gate, up, down (I x H),
    two norm gains per layer; the LM head, the final gain, one embedding row
    per sequence."""
    per_layer = 2 * nq * d * H + 2 * nkv * d * H + 3 * I * H + 2 * H
    return 2 * (L * per_layer + V * H + H + batch * H)


def test_algorithmic_bytes_match_the_shapes():
    sys.path.insert(0, str(ROOT))
    import bench
    from synth import WORKLOADS

    m8 = WORKLOADS["8b"].model
    assert bench.weight_bytes_read(m8, 1) == _hand_weight_bytes(32, 4096, 32, 8, 128, 14336, 128256, 1)
    assert bench.weight_bytes_read(m8, 1) == 15_009_857_536  # 15.010 GB, 436.2 MB per layer
    m1 = WORKLOADS["1b"].model
    assert bench.weight_bytes_read(m1, 1) == _hand_weight_bytes(16, 2048, 32, 8, 64, 8192, 128256, 1)
    assert bench.weight_bytes_read(m1, 1) == 2_471_632_896  # 2.4716 GB (tied: the LM head is the embedding)
    m70 = WORKLOADS["70b"].model
    assert bench.weight_bytes_read(m70, 16) == _hand_weight_bytes(80, 8192, 64, 8, 128, 28672, 128256, 16)
    # K and V of one cached token over every layer: 128 KB (8B), 32 KB (1B), 320 KB (70B)
    for m, per_tok in ((m8, 131072), (m1, 32768), (m70, 327680)):
        for B in (1, 8):
            assert bench.step_bytes(m, B, 101) - bench.step_bytes(m, B, 100) == B * per_tok
        # a step at context 1 (empty cache) writes the new K/V and the fp32 logits only
        assert bench.step_bytes(m, 2, 1) == bench.weight_bytes_read(m, 2) + 2 * (per_tok + m.vocab * 4)


def test_cpu_baseline_reports_the_threads_the_oracle_ran_with():
    r = _run({"OMP_NUM_THREADS": "2"})
    assert r.returncode == 0, r.stderr
    d = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
    assert d["cpu_baseline"]["cores"] == 2


def test_cpu_baseline_times_whole_oracle_steps_on_all_cores_and_one_thread():
    """Whole decode steps (every layer and the full LM head), not extrapolated
    samples: the step count asked for, on the default team and on one thread."""
    sys.path.insert(0, str(ROOT))
    import bench
    import oracle
    from synth import WORKLOADS

    m = WORKLOADS["tiny"].model
    ms, threads, model = bench.oracle_steps(m, 40, 3)
    assert len(ms) == 3 and all(t > 0 for t in ms) and threads == oracle.num_threads()
    cb = bench.cpu_baseline(m, 40, 2, 1)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and "whole decode steps" in cb["sample"]
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert oracle.num_threads() == cb["cores"]  # the default team is restored
