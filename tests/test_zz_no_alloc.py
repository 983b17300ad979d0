"""The decode entry point for callers that cannot allocate device memory.

mp_decode_attention_static takes no scratch buffer: it uses a fixed array built into
the library. Here it is called through the C ABI twice in a row (two decode steps
with different queries and lengths) and each output is compared with the ordinary
mp_decode_attention on the same inputs, within the tolerance of the other parity
tests. The file sorts last so that a failure here does not hide the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as WL
from gpu_harness import DeviceRun, rel_l2

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as m
    return m


def test_static_scratch_decode_matches_the_scratch_buffer_decode(mp):
    wl = WL.WORKLOADS[1].replace(n_prefill=5000, steps=2, append=True)
    run = DeviceRun(mp, wl, WL.generate(wl), "cuda:0")
    assert mp.mp_decode_layout_get(run.cfg).total_bytes <= mp.MP_STATIC_SCRATCH_BYTES
    run.build()
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):
        n = wl.seq_len(step)
        run.append(n - 1)
        q = run.queries[step].contiguous()
        want = run.decode(step, n).clone()
        got = torch.full_like(want, float("nan"))
        rc = mp.call_raw("mp_decode_attention_static", ctypes.byref(run.cfg), run.tables.data_ptr(),
                         run.keys.data_ptr(), run.values.data_ptr(), n, q.data_ptr(), got.data_ptr(), stream)
        assert rc == mp.MP_OK, mp.mp_status_string(rc)
        torch.cuda.synchronize()
        assert run.status() == 0
        g, w = got.cpu().numpy(), want.cpu().numpy()
        assert np.isfinite(g).all()
        for idx in np.ndindex(*g.shape[:-1]):
            assert rel_l2(g[idx], w[idx]) < TOL, (step, idx)


def test_static_scratch_rejects_configs_beyond_its_size(mp):
    wl = WL.WORKLOADS[2]
    run_cfg = mp.make_config(layers=wl.layers, batch=wl.batch, kv_heads=wl.kv_heads, q_heads=wl.q_heads,
                             head_dim=wl.head_dim, K=wl.K, L=wl.L, n_sink=wl.n_sink, window=wl.window,
                             capacity=wl.capacity, dtype=wl.dtype, w_per_layer=True)
    assert mp.mp_decode_layout_get(run_cfg).total_bytes > mp.MP_STATIC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = mp.call_raw("mp_decode_attention_static", ctypes.byref(run_cfg), fake, fake, fake, 100, fake, fake, None)
    assert rc == mp.MP_ERR_SCRATCH
