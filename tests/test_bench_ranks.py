"""The multi-process host logic of bench.py on CPU (gloo, world size 2): the
barrier and the max over ranks that the replica runs time with, and the
reference arm printing one line from rank 0 only."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks("gloo")
    r.barrier()
    got = r.max(float(10 * rank + 3))
    r.barrier()
    r.close()
    out.put((rank, got))


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 13.0, 1: 13.0}


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank0_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "flat-2^20-w4", "--steps", "1", "--warmup", "0",
                        "--gpus", "2"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 0:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
        assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    else:
        assert lines == []


def test_algorithmic_bytes_of_the_bench_workload():
    # per coordinate W*(2 g + 8 u + 8 e + 1/8 mask) + 8 theta + 8 v + 1/8 new mask,
    # per kept coordinate 8W (vals written and read) + 8 (bbar, idx)
    sys.path.insert(0, ROOT)
    import bench
    import synth
    wl = synth.WORKLOADS["llama-1.8b-w4"]
    K = 27090 * 655 + 20  # every full chunk keeps 655, the 2048-long last one 20
    b = bench.alg_bytes(wl.N, wl.W, K)["step"]
    assert K == 17_743_970
    assert abs(b - (wl.N * 88.625 + K * 40)) < 1
    assert abs(b / 1e9 - 158.052) < 0.001
