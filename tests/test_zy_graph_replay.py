"""The benchmark's launch configuration: bench.py times the whole job (build plus the
decode steps) as a replayed CUDA graph. The replay must give exactly the outputs of
the same C-ABI calls launched one by one, which the parity tests compare with the
oracle. Every stage is deterministic (integer atomics only; the split-K partials are
merged in split order), so the two runs must agree bit for bit. The file sorts last
so that a failure here does not hide the other tests."""
import os
import sys

import pytest
import torch

import workloads as WL

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as m
    return m


def test_graph_replay_gives_the_outputs_of_the_eager_calls(mp):
    import bench
    wl = WL.WORKLOADS[2].replace(name="graph-replay-1L-n8k", layers=1, n_prefill=8192, steps=4)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        job = bench.Job(mp, wl, dev, stream)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        job.run()
    torch.cuda.synchronize()
    assert (mp.mp_get_status(job.tables, stream=job.sp) & ~mp.MP_STATUS_W_NOT_BF16) == 0
    eager = job.outs.clone()
    assert torch.isfinite(eager).all()

    assert job.capture() is None
    job.outs.zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        with torch.cuda.stream(stream):
            job.run()
        torch.cuda.synchronize()
        assert (mp.mp_get_status(job.tables, stream=job.sp) & ~mp.MP_STATUS_W_NOT_BF16) == 0
        assert torch.equal(job.outs, eager)
