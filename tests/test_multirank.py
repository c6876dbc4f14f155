"""The multi-rank host logic of bench.py on CPU, world size 2 over gloo: the
job's time is the slowest rank's (MAX over ranks), its value all ranks'
FLOPs over that time, and the reference arm prints from rank 0 only.  Each
rank runs the whole workload on its own GPU (replicas: the path has no
exchange step), so nothing else crosses ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, times, out_q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_env()
        ms = bench.max_over_ranks(times[rank], got_ws)
        value = bench.whole_job_value(1e12, got_ws, ms)
        out_q.put((rank, got_ws, got_rank, got_local, ms, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    import torch.multiprocessing as mp
    ws, port = 2, _free_port()
    times = [3.0, 5.0]                                  # ms per step of each rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, times, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, got_ws, got_rank, got_local, ms, value in res:
        assert (got_ws, got_rank, got_local) == (ws, rank, rank)
        assert ms == max(times)                         # the slowest rank sets the time
        # 1e12 FLOPs per rank, two ranks, 5 ms: 400 TFLOP/s for the job
        assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_rank_passes_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.whole_job_value(2e12, 1, 4.0) == pytest.approx(500.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_from_rank0_only(rank):
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "pr1",
                        "--steps", "2", "--warmup", "0"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank != 0:
        assert lines == []
        return
    d = json.loads(lines[-1])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
