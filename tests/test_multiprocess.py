"""The N>1 path of bench.py on CPU: two gloo ranks (127.0.0.1) check the max-over-ranks
timing rule, the whole-job throughput of weak scaling (rows are independent, so each
replica takes its own batch and nothing is exchanged on the data path), and that the
reference arm's second rank exits without work."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r measured (10 + r) ms for 5 steps and a per-launch time of (1 + 2 r) ms
    got = bench.max_over_ranks([10.0 + rank, 1.0 + 2 * rank], dist, torch.device("cpu"))
    value = bench.rows_per_second(192, world, 5, got[0])
    rc = bench.run_reference(bench.parse(["--impl", "reference", "--steps", "1", "--warmup", "0"]),
                             rank, world) if rank == 1 else 0
    q.put((rank, got, value, rc))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value, rc in res:
        assert got == [11.0, 3.0]  # the max over both ranks, on every rank
        assert value == pytest.approx(192 * 2 * 5 / 0.011)
        assert rc == 0


def test_gpus_flag_plans_one_process_per_gpu():
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse(["--gpus", "2"])
    how, cmd = bench.launch_plan(a, {}, ["--gpus", "2"])
    assert how == "spawn" and "--nproc-per-node=2" in cmd and "127.0.0.1" in cmd
    assert bench.launch_plan(a, {"WORLD_SIZE": "2"}, [])[0] == "run"
    assert bench.launch_plan(a, {"WORLD_SIZE": "4"}, [])[0] == "error"
    assert bench.launch_plan(bench.parse([]), {}, [])[0] == "run"


def test_gpus_2_starts_two_replicas_of_the_reference_arm():
    """bench.py --gpus 2 without a launcher starts two ranks itself; in the reference arm
    rank 0 prints the one JSON line and rank 1 exits 0 without work (CPU only)."""
    import json
    import subprocess
    env = dict(os.environ, MASTER_PORT=str(_free_port()))
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--workload", "1", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
