"""The multi-rank host logic of bench.py, run as two gloo ranks on the CPU.

Under torchrun every rank runs the same per-GPU workload (replicas, no
data-path collective); the timed regions are bracketed by barriers, each
rank's device times are reduced element-wise with MAX, and the whole-job
value is world x per-rank work / the slowest rank's time. The reference arm
runs on rank 0 only. These are the pieces that do not need a GPU: the same
helpers run here over gloo with CPU tensors.
"""

import multiprocessing as mp
import os
import socket
import sys
import time
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2
SLEEP = 0.4


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, queue):
    try:
        if ROOT not in sys.path:
            sys.path.insert(0, ROOT)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                          WORLD_SIZE=str(WORLD))
        import torch.distributed as dist
        import bench
        dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=WORLD)
        res = {"rank": rank}
        # 1. a barrier holds every rank until the slowest arrives
        bench.barrier(WORLD)
        t0 = time.time()
        if rank == 1:
            time.sleep(SLEEP)
        bench.barrier(WORLD)
        res["waited"] = time.time() - t0
        # 2. element-wise max over ranks; every rank receives it
        mine = [0.1, 0.5, 0.25] if rank == 0 else [0.3, 0.2, 0.25]
        res["max"] = bench.max_over_ranks(mine, WORLD, "cpu")
        res["mine_after"] = mine
        # 3. the whole-job value from the slowest rank's time
        res["rate"] = bench.whole_job_rate(1e9, 10, res["max"][0], WORLD)
        # 4. the reference arm: ranks other than 0 return at once without output
        t1 = time.time()
        args = types.SimpleNamespace(steps=1, warmup=0, gpus=WORLD)
        res["ref_rc"] = bench.run_reference(args) if rank != 0 else None
        res["ref_s"] = time.time() - t1
        bench.barrier(WORLD)
        dist.destroy_process_group()
        queue.put(res)
    except Exception as e:  # reported to the parent, which fails the test
        queue.put({"rank": rank, "error": repr(e)})


@pytest.fixture(scope="module")
def results():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, queue)) for r in range(WORLD)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(WORLD):
            r = queue.get(timeout=180)
            out[r["rank"]] = r
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    for r in out.values():
        assert "error" not in r, r
    assert sorted(out) == list(range(WORLD))
    return out


def test_barrier_waits_for_slowest_rank(results):
    # rank 0 reached the second barrier at once but left it only after rank 1's sleep
    assert results[0]["waited"] >= SLEEP * 0.8
    assert results[1]["waited"] >= SLEEP


def test_max_over_ranks_is_elementwise_and_shared(results):
    for r in results.values():
        assert r["max"] == [0.3, 0.5, 0.25]
    # the input list is not changed in place
    assert results[0]["mine_after"] == [0.1, 0.5, 0.25]


def test_whole_job_value_uses_slowest_rank(results):
    # 2 ranks x 10 steps x 1e9 units, the slowest rank taking 0.3 s
    for r in results.values():
        assert r["rate"] == pytest.approx(2 * 10 * 1e9 / 0.3)


def test_reference_arm_runs_on_rank0_only(results):
    assert results[1]["ref_rc"] == 0
    assert results[1]["ref_s"] < 5.0


def test_single_rank_helpers():
    """world == 1: no process group is needed and the times come back as given."""
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([0.25, 1.5], 1, "cpu") == [0.25, 1.5]
    bench.barrier(1)
    assert bench.whole_job_rate(4.0, 3, 2.0, 1) == 6.0
