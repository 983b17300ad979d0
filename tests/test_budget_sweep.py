"""Sampled budget over the pages' (K, L) grid, with and without centering.

MagicPIG's (K, L) sweep and its centering ablation (arXiv 2410.16179v2 §4.3 "Hash function
selection" and "Data pre-processing"; the grid of Table 4 / Figure 8) relate (K, L) to
the sampled fraction of the context. For every grid point this runs the whole GPU path
on seeded cone-shaped keys (the geometry of §3.1), checks it against the fp64 oracle on
the same inputs, and prints the measured sampled fraction next to the closed-form
fraction of isotropic data (p = 1/2) and the oracle's expected fraction sum_i u_i / |R|.
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


def _expected_fraction(wl, t, centering: bool) -> float:
    """Oracle: mean over the query heads of the first KV head of sum_{i in R} u_i / |R|
    at the first decode step (u from p = 1 - theta(q, k_i - c) / pi)."""
    n = wl.seq_len(0)
    keys = t["keys"][0, 0, 0].double().numpy()
    W = t["W"][0].double().numpy()
    tab = O.HeadTables(keys, W, wl.K, wl.L, wl.n_sink, wl.n_prefill, n_total=n, centering=centering)
    lo, hi = O.lsh_region(n, wl.n_sink, wl.window)
    fr = []
    for j in range(wl.q_heads // wl.kv_heads):
        q = t["queries"][0, 0, 0, j].double().numpy()
        p = O.collision_probability(q, keys[lo:hi] - tab.center[None, :])
        fr.append(O.inclusion_probability(p, wl.K, wl.L).sum() / max(1, hi - lo))
    return float(np.mean(fr))


@pytest.mark.parametrize("K,L", GRID)
def test_budget_grid(mp, K, L):
    rows = []
    for centering in (True, False):
        wl = WL.Workload(f"sweep{K}x{L}", layers=1, batch=1, kv_heads=2, q_heads=8, head_dim=128, n_prefill=8192,
                         steps=1, append=True, K=K, L=L, dtype="bf16", seed=400 + 10 * K + L % 7)
        t = WL.generate(wl)
        rep = check_workload(mp, wl, t, centering=centering, check_csr_tables=2)
        measured = rep["sampled"] / max(1, rep["region"])
        x = 0.5 ** K
        closed = 1 - (1 - x) ** L - L * x * (1 - x) ** (L - 1)
        rows.append((centering, measured, closed, _expected_fraction(wl, t, centering)))
    for centering, measured, closed, expected in rows:
        print(f"\n[K={K} L={L} centering={'on' if centering else 'off'}] sampled={measured:.4%} "
              f"closed_form_isotropic={closed:.4%} oracle_expected={expected:.4%}")
