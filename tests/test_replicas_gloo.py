"""The N > 1 path of bench.py on the CPU: replicas only, no collective on the
data path.  Two gloo ranks each report their own step time; the job's time
is the slowest rank's, and the job's throughput counts every rank's units.
The reference arm prints from rank 0 alone."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 1.5 + rank  # rank 1 is the slower one
        ms = bench.max_over_ranks(dist, my_ms, torch.device("cpu"))
        q.put((rank, ms, bench.replica_value(1 << 20, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 2.5  # both ranks see the slowest rank's time
        assert value == pytest.approx(2 * (1 << 20) / 2.5e-3 / 1e9)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.25, None) == 3.25
    assert bench.replica_value(1 << 28, 1, 0.5) == pytest.approx((1 << 28) / 0.5e-3 / 1e9)


@pytest.mark.parametrize("rank,prints", [(0, True), (1, False)])
def test_reference_arm_prints_on_rank_0_only(rank, prints, tmp_path):
    """The oracle arm under torchrun: rank 0 runs and prints one JSON line,
    other ranks exit 0 without work (a tiny workload keeps this quick)."""
    code = (
        "import sys, types; sys.path.insert(0, %r); import bench;"
        "bench.N_FULL = 1 << 20;"
        "args = types.SimpleNamespace(steps=1, warmup=1, gpus=2);"
        "bench.run_reference(args, %d)" % (ROOT, rank))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, PYTHONPATH=ROOT))
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    if prints:
        assert len(lines) == 1
        rec = json.loads(lines[0])
        assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
        assert rec["cpu_baseline"]["kind"] == "oracle"
    else:
        assert lines == []
