"""The bench's multi-rank path on the CPU: two gloo ranks in spawned processes.

The path shards by (batch, head) problems with no exchange on the data path; across ranks there
is only the timing barrier and the max over ranks of the step time.  These tests check those
host-side pieces with world size 2: the max reduction, the barrier, the per-rank workloads (same
shape, different problems; rank 0's equal to a single-rank run's) and the whole-job value, and
that the reference arm prints nothing on a rank other than 0.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        from softmax_attention_chunk_gb300.inputs import gen_path_inputs

        ms = bench.max_over_ranks(10.0 + 5.0 * rank, ws)  # rank 1 is the slower one
        bench.barrier(ws)
        cfg = bench.rank_config(rank)
        x = gen_path_inputs(**dict(cfg, seqlen=64), heads_subset=[0])
        value = bench.job_value(1e12, ms, ws)
        out.put((rank, ms, cfg["seed"], tuple(cfg[k] for k in ("batch", "heads", "seqlen", "head_dim")),
                 x["q"].flatten()[:8].tolist(), value))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, seed0, shape0, q0, v0), (r1, ms1, seed1, shape1, q1, v1) = res
    assert (r0, r1) == (0, 1)
    assert ms0 == ms1 == 15.0                      # both ranks see the slowest rank's time
    assert shape0 == shape1 and seed0 != seed1     # weak scaling: same shape, own problems
    assert q0 != q1
    assert v0 == v1 == pytest.approx(2 * 1e12 / 15e-3 / 1e12)  # all ranks' work over the max time

    import sys

    sys.path.insert(0, ROOT)
    import bench
    from softmax_attention_chunk_gb300.inputs import gen_path_inputs

    single = gen_path_inputs(**dict(bench.rank_config(0), seqlen=64), heads_subset=[0])
    assert single["q"].flatten()[:8].tolist() == q0  # rank 0 of a 2-rank job = the 1-rank workload


def test_reference_arm_is_silent_off_rank_0(capsys, monkeypatch):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A()) is None
    assert capsys.readouterr().out == ""
