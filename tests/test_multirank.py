"""The N > 1 path of bench.py on CPU: two gloo ranks, no GPU.

The job's batch (two copies of the Llama-1B-shaped rows) is split by rows over the ranks
(tree_shard_rows); each rank plans its share with the library's planner (checked against the
oracle planner), the collectives are the max over ranks of the timings, the sum of the ranks'
tokens and the gather of the decisions on the host; the reference arm runs on rank 0 alone.
"""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    import synth
    import prefix_tree_packed_gb300 as lib
    from oracle import plan as oplan
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, qi = bench.rank_workload(2, rank, world)
        plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd, leaf1=w.leaf1, leaf2=w.leaf2)
        ref, qm = oplan.plan_forest(w.forest, max_fwd=w.max_fwd, leaf1=w.leaf1, leaf2=w.leaf2)
        t = plan.tables()
        ok = (np.array_equal(t["pos"], ref.pos) and np.array_equal(t["send"][: ref.n_tot], ref.send)
              and np.array_equal(t["r1"], qm["r1"]) and np.array_equal(t["r2"], qm["r2"]))
        q, _, _ = synth.draw_qkv(8, 8, w.hq, w.hkv, w.d, w.seed)
        # fake timings: the slower rank decides the job's time
        ms = bench.max_over_ranks(dist, [10.0 + rank, 20.0 - rank], "cpu")
        toks = bench.job_tokens(dist, plan.info.n_fwd, "cpu")
        dec = bench.gather_decisions(dist, world, qi, 1000 + qi)   # stand-in choices: the question's index
        gathered = [None] * world
        dist.all_gather_object(gathered, (float(q.astype(np.float64).sum()), ok, plan.info.n_fwd))
        out.put((rank, ms, gathered, toks, dec, len(qi)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_plan_their_own_batches_and_reduce_timings():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = [out.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, ms, gathered, toks, dec, nq in res:
        assert ms == [11.0, 20.0]                       # max over ranks, elementwise
        (s0, ok0, n0), (s1, ok1, n1) = gathered
        assert ok0 and ok1                              # each rank's native plan equals the oracle's
        assert s0 != s1                                 # different inputs on each rank
        assert n0 == n1 == 8192                         # 16 equal rows: 8 per rank
        assert toks == 16384
        assert nq == 32
        assert np.array_equal(dec, 1000 + np.arange(64))   # every question answered once, in job order
    sys.path.insert(0, ROOT)
    import bench
    # whole-job throughput: both ranks' tokens over the slowest rank's time
    assert bench.job_value(8192, 2, 10, 11.0) == pytest.approx(8192 * 2 * 10 / 0.011)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    import json
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
