"""Host logic of the multi-process benchmark on CPU (gloo, world size 2): barrier,
max-over-ranks of the timed region, and the reference arm printing on rank 0 only.
Replicas share nothing on the data path, so these are the only cross-rank steps."""
import os
import socket

import torch.multiprocessing as tmp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    r, w, _ = bench.dist_setup(use_cuda=False)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + 5.0 * r, w, use_cuda=False)
    q.put((r, w, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, 15.0), (1, 2, 15.0)]


def test_reference_arm_only_rank0_prints(monkeypatch):
    import bench
    args = type("A", (), {"workload": 0, "warmup": 0, "steps": 1})()
    assert bench.run_reference(args, rank=1, world=2) is None


def test_reference_arm_line_on_tiny_workload():
    import bench
    args = type("A", (), {"workload": 0, "warmup": 0, "steps": 1})()
    line = bench.run_reference(args, rank=0, world=1)
    assert line["impl"] == "reference" and line["unit"] == "queries/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_command_line_prints_one_json_line():
    """The command the reference arm is launched with, end to end on the CPU."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "0",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=300, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 1 and line["n_gpus"] == 1
