"""The -log u table the attention interpolates, and the cosines it does not cover.

MagicPIG (arXiv 2410.16179v2) Eq. 10/11: u = P[Binomial(L, p^K) >= T] with
p = 1 - theta/pi depends on the key only through the cosine of the hashed query with
k - c, so the table build writes -log u at 4097 cosines in [-0.5, 0.99] once per config
and the attention interpolates it; below -0.5 (u near zero) and above 0.99 (where
1 - acos(c)/pi has its square-root edge) the attention evaluates u directly. Checked
here: the stored table against the oracle's inclusion probability at every grid point,
for several (K, L, T); and full parity on heads whose query is a key's centered vector
(cosine 1 with that key: the direct branch) or its negative.

The table holds the kernel's own fp32 evaluation (acosf, log1pf, expm1f and expf of
arguments up to about L·|log(1 - x)|, a few units in the last place each), so it is
compared with the fp64 oracle within 5e-5 absolute plus 1e-4 relative; a float32 model
of the same steps stays within 1.3e-5 absolute for these configs.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from gpu_harness import DeviceRun, check_workload

pytestmark = pytest.mark.gpu

LUT_N, LUT_LO, LUT_HI = 4096, -0.5, 0.99


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as m
    return m


@pytest.mark.parametrize("K,L,T", [(10, 150, 2), (9, 120, 2), (8, 75, 1), (12, 250, 3), (6, 40, 7), (1, 1, 1),
                                   (0, 16, 2)])
def test_table_matches_the_oracle(mp, K, L, T):
    wl = WL.Workload("lut", layers=1, batch=1, kv_heads=1, q_heads=1, head_dim=64, n_prefill=300, steps=1,
                     append=False, K=K, L=L, dtype="f32", seed=5, window=8)
    run = DeviceRun(mp, wl, WL.generate(wl), "cuda:0", threshold=T)
    run.build()
    torch.cuda.synchronize()
    off = run.tl.logu_lut
    got = run.tables[off:off + 4 * (LUT_N + 1)].view(torch.float32).cpu().double().numpy()
    cs = LUT_LO + (LUT_HI - LUT_LO) * np.arange(LUT_N + 1) / LUT_N
    p = 1.0 - np.arccos(cs) / np.pi
    want = -np.log(np.maximum(O.inclusion_probability(p, K, L, T), 1e-30))
    np.testing.assert_allclose(got, want, rtol=1e-4, atol=5e-5)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_query_along_a_centered_key(mp, sign):
    """Query heads 0 and 2 of every KV head of the layer are (+/-) a key's centered vector
    (bf16-rounded), so the cosine with that key is about +/-1, outside the table."""
    wl = WL.WORKLOADS[1].replace(name="aligned-queries", n_prefill=6000, steps=3, append=True)
    t = WL.generate(wl)
    keys = t["keys"]
    for h in range(wl.kv_heads):
        c = O.center_of_keys(keys[0, 0, h].double().numpy(), wl.n_sink, wl.n_prefill)
        for s in range(wl.steps):
            for j, qh in ((1000 + 7 * h, h * wl.group), (4000 + 11 * h, h * wl.group + 2)):
                kc = keys[0, 0, h, j].double().numpy() - c
                t["queries"][s, 0, 0, qh] = torch.from_numpy(sign * 4.0 * kc / np.linalg.norm(kc)).to(t["queries"].dtype)
    rep = check_workload(mp, wl, t, check_csr_tables=4)
    assert rep["heads"] == wl.q_heads * wl.steps


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_keys_at_every_cosine_with_the_query(mp, dtype):
    """Keys placed at prescribed cosines a in [-0.95, 0.998] with the query around a
    common point, with K = 1, L = 4, T = 1 so that even keys at a = -0.9 (p = 0.14) are
    sampled often: the sampled set holds keys on both sides of the table's range and
    inside it, and the output must match the oracle."""
    wl = WL.Workload("cosines", layers=1, batch=1, kv_heads=1, q_heads=1, head_dim=64, n_prefill=2000, steps=1,
                     append=False, K=1, L=4, dtype=dtype, seed=77, window=8)
    t = WL.generate(wl)
    rng = np.random.default_rng(77)
    d, n = wl.head_dim, wl.capacity
    q = rng.standard_normal(d)
    qh = q / np.linalg.norm(q)
    c0 = 3.0 * rng.standard_normal(d)
    a = rng.uniform(-0.95, 0.998, n)
    a[::50] = 0.996  # some keys above the table's range for sure
    r = rng.standard_normal((n, d))
    r -= np.outer(r @ qh, qh)
    r /= np.linalg.norm(r, axis=1, keepdims=True)
    keys = c0 + 5.0 * (a[:, None] * qh + np.sqrt(1 - a[:, None] ** 2) * r)
    t["keys"][0, 0, 0] = torch.from_numpy(keys).to(t["keys"].dtype)
    t["queries"][0, 0, 0, 0] = torch.from_numpy(2.0 * q).to(t["queries"].dtype)
    k64 = t["keys"][0, 0, 0].double().numpy()
    kc = k64 - O.center_of_keys(k64, wl.n_sink, wl.n_prefill)
    qq = t["queries"][0, 0, 0, 0].double().numpy()
    cos = kc @ qq / np.linalg.norm(kc, axis=1) / np.linalg.norm(qq)
    assert (cos < LUT_LO).sum() > 200 and (cos > LUT_HI).sum() > 20  # both sides of the table occur
    rep = check_workload(mp, wl, t, threshold=1, check_csr_tables=wl.L)
    assert rep["heads"] == 1 and rep["sampled"] > 1000
