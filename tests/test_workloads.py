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


def test_tight_cone_and_constant_keys():
    """The tight-cone recipe puts the keys at cosine ~a/sqrt(a^2 + d) from mu and the sink
    at -sink_scale·a·mu; constant keys are a·mu exactly."""
    wl = WL.WORKLOADS[1].replace(cone=40.0, sink_scale=1.0)
    mu = WL.head_mu(wl, 0, 0, 5)
    k = WL.keys_block(wl, 0, 0, 5, 0, 4000)
    assert torch.allclose(k[0], -40.0 * mu)
    cos = (k[1:] @ mu) / torch.linalg.vector_norm(k[1:], dim=1)
    assert abs(cos.mean().item() - 40.0 / math.sqrt(40.0 ** 2 + 128)) < 0.01
    # pairwise cosine of two keys: about a^2 / (a^2 + d)
    kk = k[1:2001] / torch.linalg.vector_norm(k[1:2001], dim=1, keepdim=True)
    pair = (kk[:1000] * kk[1000:]).sum(dim=1).mean().item()
    assert abs(pair - 1600.0 / (1600.0 + 128)) < 0.01
    c = WL.keys_block(wl.replace(constant_keys=True), 0, 0, 5, 0, 50)
    assert torch.equal(c[1:], (40.0 * mu)[None, :].expand(49, -1))
    assert torch.allclose(c[0], -40.0 * mu)


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


def _generate_block_by_block(wl):
    """The tensors of generate() assembled from the one-block functions."""
    cap, d = wl.capacity, wl.head_dim
    keys = torch.zeros(wl.layers, wl.batch, wl.kv_heads, cap, d, dtype=wl.torch_dtype)
    values = torch.zeros_like(keys)
    queries = torch.zeros(wl.steps, wl.layers, wl.batch, wl.q_heads, d, dtype=wl.torch_dtype)
    for l in range(wl.layers):
        for b in range(wl.batch):
            for h in range(wl.kv_heads):
                keys[l, b, h] = WL.round_to(WL.keys_block(wl, l, b, h, 0, cap), wl.dtype)
                values[l, b, h] = WL.round_to(WL.values_block(wl, l, b, h, 0, cap), wl.dtype)
            for s in range(wl.steps):
                queries[s, l, b] = WL.round_to(WL.query_block(wl, s, l, b), wl.dtype)
    return keys, values, queries


def test_generate_equals_the_block_functions():
    """generate() draws all heads and steps of a sequence at once; every element must be
    the one the single-block functions give."""
    cases = [WL.WORKLOADS[0],
             WL.Workload("mix", layers=2, batch=2, kv_heads=3, q_heads=6, head_dim=128, n_prefill=1037,
                         steps=5, append=True, K=6, L=20, dtype="bf16", seed=17, iso_fraction=0.1,
                         w_per_layer=True),
             WL.WORKLOADS[1].replace(n_prefill=3000, steps=3),
             WL.WORKLOADS[1].replace(n_prefill=700, steps=2, cone=40.0, sink_scale=1.0),
             WL.WORKLOADS[0].replace(n_prefill=300, constant_keys=True)]
    for wl in cases:
        t = WL.generate(wl)
        k, v, q = _generate_block_by_block(wl)
        assert torch.equal(t["keys"], k), wl.name
        assert torch.equal(t["values"], v), wl.name
        assert torch.equal(t["queries"], q), wl.name


def test_stream_draws_equal_single_stream_draws():
    keys = [WL.stream_key(5, i) for i in range(4)]
    g = WL.gaussian_streams(keys, 1000, offset=77)
    u = WL.uniform_streams(keys, 333, offset=5)
    for i, key in enumerate(keys):
        assert torch.equal(g[i], WL.gaussian(key, 1000, offset=77))
        assert torch.equal(u[i], WL.uniform(key, 333, offset=5))
