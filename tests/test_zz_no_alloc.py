"""The decode entry point for callers that cannot allocate device memory.

mp_decode_attention_static takes no scratch buffer: it uses a fixed array built into
the library. Here it is called through the C ABI several times in a row (decode steps
with different queries and lengths, a long one before a short one so that the array
still holds the longer call's lists and partials) and each output is compared with the
ordinary mp_decode_attention on the same inputs. Both run the same kernels, whose
results do not depend on scheduling (integer atomics only, split-K partials merged in
split order), so the outputs must agree bit for bit; one step is also checked against
the oracle. The file sorts last so that a failure here does not hide the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
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


def _static(mp, run, n, q, out):
    stream = torch.cuda.current_stream().cuda_stream
    return mp.call_raw("mp_decode_attention_static", ctypes.byref(run.cfg), run.tables.data_ptr(),
                       run.keys.data_ptr(), run.values.data_ptr(), n, q.data_ptr(), out.data_ptr(), stream)


def test_static_scratch_decode_matches_the_scratch_buffer_decode(mp):
    wl = WL.WORKLOADS[1].replace(n_prefill=5000, steps=3, append=True)
    t = WL.generate(wl)
    run = DeviceRun(mp, wl, t, "cuda:0")
    assert mp.mp_decode_layout_get(run.cfg).total_bytes <= mp.MP_STATIC_SCRATCH_BYTES
    run.build()
    # (step, n): two appending steps, then the third step's query over a shorter prefix
    # (the lists, partials and counters of the longer calls are still in the array)
    calls = [(0, wl.seq_len(0)), (1, wl.seq_len(1)), (2, 2345)]
    for step, n in calls:
        if step < 2:
            run.append(n - 1)
        q = run.queries[step].contiguous()
        want = run.decode(step, n).clone()
        got = torch.full_like(want, float("nan"))
        rc = _static(mp, run, n, q, got)
        assert rc == mp.MP_OK, mp.mp_status_string(rc)
        torch.cuda.synchronize()
        assert run.status() == 0
        assert torch.isfinite(got).all()
        assert torch.equal(got, want), (step, n)
        g, w = got.cpu().numpy(), want.cpu().numpy()
        for idx in np.ndindex(*g.shape[:-1]):
            assert rel_l2(g[idx], w[idx]) < TOL, (step, idx)
        if step == 2:
            # one KV head of the short call against the oracle (its own codes end to end)
            k = t["keys"][0, 0, 3, :n].double().numpy()
            v = t["values"][0, 0, 3, :n].double().numpy()
            tab = O.HeadTables(t["keys"][0, 0, 3].double().numpy(), t["W"][0].double().numpy(), wl.K, wl.L,
                               wl.n_sink, wl.n_prefill)
            for j in range(12, 16):
                r = O.decode_head(t["queries"][step, 0, 0, j].double().numpy(), k, v, tab, n, wl.window)
                assert rel_l2(g[0, 0, j], r["out"]) < TOL, j


def test_static_scratch_rejects_configs_beyond_its_size(mp):
    wl = WL.WORKLOADS[2]
    run_cfg = mp.make_config(layers=wl.layers, batch=wl.batch, kv_heads=wl.kv_heads, q_heads=wl.q_heads,
                             head_dim=wl.head_dim, K=wl.K, L=wl.L, n_sink=wl.n_sink, window=wl.window,
                             capacity=wl.capacity, dtype=wl.dtype, w_per_layer=True)
    assert mp.mp_decode_layout_get(run_cfg).total_bytes > mp.MP_STATIC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = mp.call_raw("mp_decode_attention_static", ctypes.byref(run_cfg), fake, fake, fake, 100, fake, fake, None)
    assert rc == mp.MP_ERR_SCRATCH
