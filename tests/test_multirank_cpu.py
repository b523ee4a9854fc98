"""The N>1 bench path on CPU: two gloo ranks, each with its own replica of the
work, reduce to (max elapsed, summed units) exactly as bench.py does."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed, units = bench.reduce_over_ranks(1.5 + rank, 10.0 * (rank + 1), dist)
    q.put((rank, elapsed, units))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.0, 7.0, None) == (3.0, 7.0)


def test_reference_arm_prints_the_contract_line(capsys):
    # the reference arm is the CPU oracle: it runs here, on a bounded sample per step
    import json
    import bench
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 3 and line["value"] > 0
    assert line["config"]["workload"] == bench.WORKLOAD and line["config"]["heads"] == 64
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_bench_rejects_fewer_than_three_warmup_steps():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--steps", "1", "--warmup", "2"])


def test_gpus_n_without_torchrun_starts_n_ranks():
    # --gpus 2 with no torchrun environment: bench.py starts both ranks itself;
    # the reference arm runs on rank 0 and reports the world size
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_replica_count_covers_l2():
    import bench
    # copies whose step inputs together cover three L2s, clamped to [2, 64]
    l2 = 126 * 2 ** 20
    for per in (7.3e6, 30e6, 151e6, 1e9):
        n = bench.replica_count(per, l2)
        assert 2 <= n <= 64
        if n < 64:
            assert n * per >= 3 * l2 and (n == 2 or (n - 1) * per < 3 * l2)
    assert bench.replica_count(1, l2) == 64 and bench.replica_count(1e12, l2) == 2
