"""Sampled budget over the pages' (K, L) grid, with and without centering.

MagicPIG's (K, L) sweep and its centering ablation (arXiv 2410.16179v2 §4.3 "Hash function
selection" and "Data pre-processing"; the grid of Table 4 / Figure 8) relate (K, L) to
the sampled fraction of the context. For every grid point this runs the whole GPU path
on seeded cone-shaped keys (the geometry of §3.1), checks it against the fp64 oracle on
the same inputs, and checks the GPU's sampled count against the oracle's expected count
sum_i u_i (printing both next to the closed-form fraction of isotropic data, p = 1/2).
"""
import numpy as np
import pytest
import torch

import workloads as WL
from oracle import magicpig_oracle as O

from gpu_harness import check_workload

pytestmark = pytest.mark.gpu

GRID = [(8, 75), (8, 90), (9, 120), (10, 150), (10, 220), (10, 300), (11, 300)]


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as m
    return m


def _expected_budget(wl, t, centering: bool):
    """Oracle: sum over every query head of the first decode step of sum_{i in R} u_i and
    of u_i (1 - u_i), with u from p = 1 - theta(q, k_i - c) / pi: the expected sampled
    count over the draws of W and its binomial variance."""
    n = wl.seq_len(0)
    lo, hi = O.lsh_region(n, wl.n_sink, wl.window)
    W = t["W"][0].double().numpy()
    su = var = 0.0
    for h in range(wl.kv_heads):
        keys = t["keys"][0, 0, h].double().numpy()
        tab = O.HeadTables(keys, W, wl.K, wl.L, wl.n_sink, wl.n_prefill, n_total=n, centering=centering)
        for j in range(wl.group):
            q = t["queries"][0, 0, 0, h * wl.group + j].double().numpy()
            p = O.collision_probability(q, keys[lo:hi] - tab.center[None, :])
            u = O.inclusion_probability(p, wl.K, wl.L)
            su += float(u.sum())
            var += float((u * (1.0 - u)).sum())
    return su, var, wl.q_heads * (hi - lo)


# Bound on |S| - sum u in binomial standard deviations. For one W the sampling events of
# different keys and query heads are positively correlated (keys at similar angles share
# their buckets), so the spread is wider than the binomial one: on these seeded inputs
# the oracle's own |S| lies between -1.5 and +3.8 binomial deviations from sum u.
BUDGET_SIGMAS = 6.0


@pytest.mark.parametrize("K,L", GRID)
def test_budget_grid(mp, K, L):
    """The GPU's sampled count over all query heads against the oracle's expected count
    sum_i u_i (the budget relation of the (K, L) choice), centering on and off."""
    rows = []
    for centering in (True, False):
        wl = WL.Workload(f"sweep{K}x{L}", layers=1, batch=1, kv_heads=2, q_heads=8, head_dim=128, n_prefill=8192,
                         steps=1, append=True, K=K, L=L, dtype="bf16", seed=400 + 10 * K + L % 7)
        t = WL.generate(wl)
        rep = check_workload(mp, wl, t, centering=centering, check_csr_tables=2)
        su, var, region = _expected_budget(wl, t, centering)
        assert rep["region"] == region
        x = 0.5 ** K
        closed = 1 - (1 - x) ** L - L * x * (1 - x) ** (L - 1)
        z = (rep["sampled"] - su) / np.sqrt(var)
        rows.append((centering, rep["sampled"], su, z, closed, region))
        assert abs(z) < BUDGET_SIGMAS, (K, L, centering, rep["sampled"], su, z)
    for centering, sampled, su, z, closed, region in rows:
        print(f"\n[K={K} L={L} centering={'on' if centering else 'off'}] sampled={sampled / region:.4%} "
              f"oracle_expected={su / region:.4%} z={z:+.2f} closed_form_isotropic={closed:.4%}")
