"""Host-side logic of bench.py: the reference arm (the CPU oracle), the replica
reductions of the N > 1 path over gloo (world size 2, CPU), and the JSON helpers."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ENV = dict(os.environ, MASTER_ADDR="127.0.0.1", OMP_NUM_THREADS="2")


def _json_lines(out):
    return [json.loads(ln) for ln in out.splitlines() if ln.startswith("{")]


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--cpu-budget", "0.05"], cwd=ROOT, capture_output=True, text=True, env=ENV, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    (line,) = _json_lines(r.stdout)
    assert line["impl"] == "reference" and line["unit"] == "GPoints/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["workload"] == "star25_lap8_512"


def test_reference_arm_two_ranks_gloo():
    """Under torchrun with two ranks only rank 0 runs and prints; the other exits 0."""
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                        "--master-addr", "127.0.0.1", "--master-port", "29531", "bench.py", "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.05"],
                       cwd=ROOT, capture_output=True, text=True, env=ENV, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference"


def _reduce_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, local, w = bench.dist_setup(world)
    bench.barrier(dist)
    mx = bench.max_over_ranks(dist, float(rank + 1) * 10.0)
    sm = bench.sum_over_ranks(dist, float(rank + 1))
    q.put((rank, w, mx, sm))
    dist.destroy_process_group()


def test_replica_reductions_over_gloo():
    """The N > 1 timing rule: max of the ranks' times, sum of the ranks' work."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_reduce_worker, args=(r, 2, 29533, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 20.0, 3.0), (1, 2, 20.0, 3.0)]


def test_json_helpers():
    sys.path.insert(0, ROOT)
    import bench
    peak, kind = bench.peaks()
    assert peak > 1000 and kind in ("measured", "fallback")
    h = bench.kernel_source_hash()
    assert len(h) == 16
    t = bench.profiled_traffic("star25_512")
    assert t is None or t > 1e9
    # The recorded traffic is reported only for the launch geometry it was captured on.
    e = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["star25_512"]
    if t is not None:
        assert bench.profiled_traffic("star25_512", dict(e["launch"])) == t
        assert bench.profiled_traffic("star25_512", dict(e["launch"], zchunks=e["launch"]["zchunks"] + 1)) is None
