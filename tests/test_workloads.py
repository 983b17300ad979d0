"""Host-side checks of the seeded synthetic input generator."""
import math

import torch

import workloads as WL


def test_counter_generator_is_blockwise_consistent():
    wl = WL.WORKLOADS[1]
    full = WL.keys_block(wl, 0, 0, 3, 0, 300)
    part = WL.keys_block(wl, 0, 0, 3, 120, 300)
    assert torch.equal(full[120:], part)
    assert torch.equal(full[:5], WL.keys_block(wl, 0, 0, 3, 0, 5))
    v = WL.values_block(wl, 0, 0, 3, 7, 9)
    assert torch.equal(v, WL.values_block(wl, 0, 0, 3, 0, 9)[7:])


def test_gaussian_moments_and_independence_of_streams():
    g = WL.gaussian(WL.stream_key(1, 2, 3), 400000)
    assert abs(g.mean().item()) < 5 / math.sqrt(4e5)
    assert abs(g.var().item() - 1) < 0.01
    h = WL.gaussian(WL.stream_key(1, 2, 4), 400000)
    assert abs(torch.corrcoef(torch.stack([g, h]))[0, 1].item()) < 0.01


def test_cone_geometry_of_keys_and_queries():
    wl = WL.WORKLOADS[1]
    mu = WL.head_mu(wl, 0, 0, 2)
    k = WL.keys_block(wl, 0, 0, 2, 0, 2000)
    assert torch.allclose(k[0], -6 * mu)
    assert abs((k[1:] @ mu).mean().item() - 3.0) < 0.1
    q = WL.query_block(wl, 0, 0, 0)
    assert abs((q[8:12] @ mu).mean().item() + 2.0) < 2.0


def test_generate_shapes_and_dtypes():
    wl = WL.WORKLOADS[0]
    t = WL.generate(wl)
    assert t["keys"].shape == (1, 1, 1, 2048, 64) and t["keys"].dtype == torch.float32
    assert t["W"].shape == (1, 64, 600)
    assert t["queries"].shape == (1, 1, 1, 1, 64)
    small = wl.replace(dtype="bf16", w_bf16=True, n_prefill=40)
    t2 = WL.generate(small)
    assert t2["keys"].dtype == torch.bfloat16
    assert torch.equal(t2["W"].to(torch.bfloat16).to(torch.float32), t2["W"])


def test_isotropic_mix_fraction():
    wl = WL.WORKLOADS[4]
    mu = WL.head_mu(wl, 0, 1, 0)
    k = WL.keys_block(wl, 0, 1, 0, 1, 20001)
    frac = ((k @ mu) < 1.0).double().mean().item()   # cone keys sit near 3 along mu
    assert 0.08 < frac < 0.13
