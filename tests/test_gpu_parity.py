"""GPU parity: the CUDA path through the C ABI against the CPU oracle, stage by stage
(codes, bucket tables, query codes, sampled sets, exact tokens, outputs) on seeded
synthetic workloads. Codes are compared bit-exactly except near-tie projections
(|y| < 1e-5 ||x|| ||w_j||), which are counted; sampled sets exactly on the GPU's
codes; outputs within 2e-3 relative L2 of the fp64 oracle."""
import numpy as np
import pytest
import torch

import workloads as WL
from gpu_harness import DeviceRun, check_workload, config_for, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as m
    return m


def _report(name, rep):
    print(f"\n[{name}] mode={'csr' if rep['match_mode'] == 1 else 'scan'} heads={rep['heads']} max_rel_l2={rep['max_rel_l2']:.2e} "
          f"sampled_frac={rep['sampled'] / max(1, rep['region']):.4f} codes_differ(near-tie)={rep['codes_differ']} "
          f"q_codes_differ(near-tie)={rep['q_codes_differ']} S_differ_vs_oracle_codes={rep['S_differ_oracle_codes']}")


def test_config0_tiny_fp32(mp):
    wl = WL.WORKLOADS[0]
    rep = check_workload(mp, wl, WL.generate(wl), check_csr_tables=wl.L)
    _report("cfg0", rep)
    assert rep["heads"] == 1


def test_config1_llama8b_layer(mp):
    wl = WL.WORKLOADS[1]
    rep = check_workload(mp, wl, WL.generate(wl), check_csr_tables=8)
    _report("cfg1", rep)
    assert rep["heads"] == 32


RAGGED = WL.Workload("ragged-appends", layers=2, batch=2, kv_heads=2, q_heads=8, head_dim=128,
                     n_prefill=1037, steps=40, append=True, K=6, L=20, dtype="bf16", seed=17, window=16,
                     w_per_layer=True)


def test_ragged_appends_leave_the_window(mp):
    """Appended tokens leave the window after 16 steps and are then matched from
    the stored codes; prefill length not a multiple of any tile."""
    rep = check_workload(mp, RAGGED, WL.generate(RAGGED), steps=[0, 15, 16, 17, 39], check_csr_tables=20)
    _report("ragged", rep)


@pytest.mark.parametrize("kw", [
    dict(dtype="f32", head_dim=128, w_bf16=False),
    dict(dtype="bf16", head_dim=64),
    dict(dtype="bf16", head_dim=128, w_bf16=False),   # fp32 W: three-term bf16 split on the tensor cores
    dict(dtype="bf16", head_dim=64, w_bf16=False),
    dict(dtype="f32", head_dim=64, q_heads=2, kv_heads=2, w_bf16=False),
])
def test_dtypes_and_head_dims(mp, kw):
    wl = WL.Workload("dt", layers=1, batch=1, kv_heads=2, q_heads=4, head_dim=128, n_prefill=2500, steps=2,
                     append=True, K=7, L=30, dtype="bf16", seed=23).replace(**kw)
    rep = check_workload(mp, wl, WL.generate(wl))
    _report(str(kw), rep)


@pytest.mark.parametrize("mode", [1, 2])
def test_centering_off(mp, mode):
    """The pages' centering ablation: keys hashed as they are (c = 0), p from cos(q, k),
    in both match modes; the cone-shaped keys then give a different sampled budget."""
    wl = WL.Workload("nocenter", layers=1, batch=1, kv_heads=2, q_heads=8, head_dim=128, n_prefill=6000,
                     steps=3, append=True, K=8, L=60, dtype="bf16", seed=77)
    t = WL.generate(wl)
    off = check_workload(mp, wl, t, match_mode=mode, centering=False, check_csr_tables=wl.L)
    _report("centering off", off)
    on = check_workload(mp, wl, t, match_mode=mode, check_csr_tables=4)
    _report("centering on", on)
    assert off["sampled"] != on["sampled"]


@pytest.mark.parametrize("threshold,mode", [(1, 1), (1, 2), (3, 1), (3, 2), (5, 1), (7, 2)])
def test_thresholds(mp, threshold, mode):
    """u = P[Bin(L, p^K) >= T] and the sampling rule for T other than the pages' 2
    (a reviewer's question in the authors' responses), in both match modes."""
    wl = WL.Workload(f"t{threshold}", layers=1, batch=1, kv_heads=2, q_heads=4, head_dim=128, n_prefill=3000,
                     steps=20, append=True, K=6, L=40, dtype="bf16", seed=31 + threshold, window=8)
    rep = check_workload(mp, wl, WL.generate(wl), threshold=threshold, match_mode=mode, steps=[0, 19],
                         check_csr_tables=wl.L)
    _report(f"threshold {threshold}", rep)
    assert rep["match_mode"] == mode


def test_K0_samples_everything_and_equals_exact_attention(mp):
    wl = WL.Workload("k0", layers=1, batch=1, kv_heads=1, q_heads=2, head_dim=128, n_prefill=700, steps=1,
                     append=False, K=0, L=3, dtype="bf16", seed=5)
    t = WL.generate(wl)
    rep = check_workload(mp, wl, t)
    assert rep["sampled"] == rep["region"]
    run = DeviceRun(mp, wl, t, "cuda:0")
    run.build()
    out = run.decode(0, 700).cpu().numpy()
    k = t["keys"][0, 0, 0].double().numpy()
    v = t["values"][0, 0, 0].double().numpy()
    for j in range(2):
        q = t["queries"][0, 0, 0, j].double().numpy()
        lg = k @ q / np.sqrt(128)
        e = np.exp(lg - lg.max())
        assert rel_l2(out[0, 0, j], e @ v / e.sum()) < 2e-3


def test_short_sequences_are_all_exact(mp):
    wl = WL.Workload("short", layers=1, batch=2, kv_heads=1, q_heads=1, head_dim=64, n_prefill=3, steps=70,
                     append=True, K=5, L=8, dtype="bf16", seed=9)
    rep = check_workload(mp, wl, WL.generate(wl), steps=[0, 1, 60, 66, 67, 69])
    _report("short", rep)


def test_status_flags(mp):
    wl = WL.Workload("st", layers=1, batch=1, kv_heads=1, q_heads=1, head_dim=128, n_prefill=300, steps=100,
                     append=True, K=4, L=4, dtype="bf16", seed=3, window=8)
    t = WL.generate(wl)
    run = DeviceRun(mp, wl, t, "cuda:0")
    # decode on never-built tables
    run.tables.zero_()
    run.decode(0, 300)
    assert run.status() & mp.MP_STATUS_NOT_BUILT
    # W that bf16 cannot hold exactly
    run.W += 1e-3 * torch.randn_like(run.W)
    run.build()
    assert run.status() == mp.MP_STATUS_W_NOT_BF16
    # a clean build, then a decode that needs codes of tokens never appended
    run.W.copy_(t["W"].to(run.W.device))
    run.build()
    run.decode(0, 300)
    assert run.status() == 0
    run.decode(0, 350)
    assert run.status() == mp.MP_STATUS_APPEND_GAP


@pytest.mark.parametrize("path,w_bf16", [("simt", True), ("tc", True), ("simt", False), ("tc", False)])
def test_both_key_hash_paths_match_the_oracle(mp, path, w_bf16, monkeypatch):
    """Keys, queries and appended keys are hashed on tensor cores (default) or on CUDA
    cores (MP_HASH_PATH=simt); both must give the oracle's codes except near ties, with
    one W per layer, bf16-representable or not (three-term split on the tensor cores)."""
    monkeypatch.setenv("MP_HASH_PATH", path)
    wl = WL.Workload("paths", layers=2, batch=1, kv_heads=2, q_heads=4, head_dim=128, n_prefill=4099, steps=2,
                     append=True, K=10, L=50, dtype="bf16", seed=41, w_per_layer=True, w_bf16=w_bf16)
    rep = check_workload(mp, wl, WL.generate(wl), check_csr_tables=50)
    _report(f"hash path {path}", rep)


@pytest.mark.parametrize("K,L,d", [(9, 120, 128), (12, 40, 128), (7, 33, 64), (1, 5, 64), (12, 1024, 128)])
def test_tensor_core_hash_tile_layouts(mp, K, L, d):
    """Tables per 256-column tile = floor(256/K): K values that leave padding columns,
    L not a multiple of it, both head dims; the largest K and L the library takes."""
    wl = WL.Workload(f"tc-{K}-{L}-{d}", layers=1, batch=1, kv_heads=1, q_heads=2, head_dim=d, n_prefill=700,
                     steps=1, append=False, K=K, L=L, dtype="bf16", seed=K * 100 + L)
    rep = check_workload(mp, wl, WL.generate(wl), check_csr_tables=L)
    _report(f"tc K={K} L={L} d={d}", rep)


def test_maximum_capacity(mp):
    """The largest capacity the library takes, 2^19 tokens, filled by the prefill up to
    the two appended tokens: 16 bucketed segments per table (the last one ragged), the
    match kernel's per-token bitmaps at their largest, and ~10^4 sampled keys per head
    split across many attention slices."""
    wl = WL.Workload("max-capacity", layers=1, batch=1, kv_heads=1, q_heads=4, head_dim=128,
                     n_prefill=(1 << 19) - 2, steps=2, append=True, K=8, L=32, dtype="bf16", seed=19)
    assert wl.capacity == 1 << 19
    assert mp.mp_config_check(config_for(mp, wl)) == mp.MP_OK
    assert mp.mp_config_check(config_for(mp, wl.replace(n_prefill=(1 << 19) - 1))) == mp.MP_ERR_UNSUPPORTED
    rep = check_workload(mp, wl, WL.generate(wl), check_csr_tables=4)
    _report("max capacity", rep)
    assert rep["match_mode"] == mp.MP_MATCH_CSR and rep["heads"] == 8


# ----------------------------------------------------------------------------------
# full-size workloads, same ABI calls as the benchmark; the oracle checks sampled
# KV heads (all their query heads) at the first and last decode steps
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("cfg,units,steps", [
    (2, [(0, 0, 0), (31, 0, 7)], [0, 63]),
    (3, [(0, 0, 0), (0, 15, 39)], [0, 31]),
    (4, [(0, 0, 0), (0, 3, 7)], [0, 63]),
])
def test_full_size_workloads_sampled(mp, cfg, units, steps):
    wl = WL.WORKLOADS[cfg]
    t = WL.generate(wl, device="cuda")
    torch.cuda.synchronize()
    rep = check_workload(mp, wl, t, units=units, steps=steps, check_csr_tables=6)
    _report(f"cfg{cfg} full size (sampled)", rep)
    assert rep["heads"] == len(units) * wl.group * len(steps)
    del t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("wl", [
    WL.WORKLOADS[1].replace(kv_heads=4, q_heads=16, n_prefill=6000),
    RAGGED,
    WL.Workload("scan-mha-t1", layers=1, batch=2, kv_heads=3, q_heads=3, head_dim=64, n_prefill=2222, steps=3,
                append=True, K=5, L=17, dtype="f32", seed=77, w_bf16=False),
    WL.Workload("scan-g16", layers=1, batch=1, kv_heads=1, q_heads=16, head_dim=128, n_prefill=3000, steps=1,
                append=False, K=4, L=24, dtype="bf16", seed=78),
], ids=["cfg1-like", "ragged", "mha-f32", "group16"])
def test_scan_match_mode(mp, wl):
    """Bit-plane streaming match, forced (and chosen by AUTO for small K / large groups)."""
    steps = [0, 15, 16, 17, 39] if wl is RAGGED else None
    rep = check_workload(mp, wl, WL.generate(wl), match_mode=mp.MP_MATCH_SCAN, steps=steps,
                         check_csr_tables=wl.L)
    _report(f"scan {wl.name}", rep)
    assert rep["match_mode"] == mp.MP_MATCH_SCAN


# ----------------------------------------------------------------------------------
# mp_decode_step: the append and the decode of a step in one call, the appended keys
# and the queries hashed by one launch
# ----------------------------------------------------------------------------------

STEP_CASES = {
    "gqa4": WL.WORKLOADS[1].replace(n_prefill=5000, steps=20, append=True, window=8),
    "gqa8-b4": WL.WORKLOADS[4].replace(n_prefill=4000, steps=12, window=8),       # two row blocks per layer
    "mha-b16": WL.WORKLOADS[3].replace(n_prefill=3000, steps=3, window=8),        # five row blocks per layer
    "ragged": RAGGED,
}


@pytest.mark.parametrize("case,path,kw", [
    ("gqa4", "tc", {}), ("gqa4", "simt", {}), ("gqa4", "tc", dict(center_query=True)),
    ("gqa8-b4", "tc", {}), ("gqa8-b4", "tc", dict(center_query=True)), ("mha-b16", "tc", {}),
    ("ragged", "tc", {}), ("ragged", "tc", dict(w_bf16=False)), ("ragged", "tc", dict(match_mode=2)),
    ("gqa4", "tc", dict(K=0, L=3)),
])
def test_decode_step_equals_append_then_decode(mp, monkeypatch, case, path, kw):
    """Same codes, query codes, lists and outputs, bit for bit, as the two separate calls."""
    monkeypatch.setenv("MP_HASH_PATH", path)
    kw = dict(kw)
    cq = kw.pop("center_query", False)
    mode = kw.pop("match_mode", 0)
    wl = STEP_CASES[case].replace(**kw)
    t = WL.generate(wl)
    a = DeviceRun(mp, wl, t, "cuda:0", match_mode=mode, center_query=cq)
    b = DeviceRun(mp, wl, t, "cuda:0", match_mode=mode, center_query=cq)
    a.build()
    b.build()
    for step in range(wl.steps):
        n = wl.seq_len(step)
        a.append(n - 1)
        oa = a.decode(step, n).clone()
        ob = b.step(step, n).clone()
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), (case, step)
        qa, la, sa = a.decode_state()
        qb, lb, sb = b.decode_state()
        np.testing.assert_array_equal(qa, qb)
        np.testing.assert_array_equal(la, lb)
        np.testing.assert_array_equal(sa, sb)
        if step in (0, wl.steps - 1):
            for qi in range(len(la)):
                np.testing.assert_array_equal(a.list_of(qi, int(la[qi])), b.list_of(qi, int(lb[qi])))
    assert (a.status() & ~mp.MP_STATUS_W_NOT_BF16) == 0 and (b.status() & ~mp.MP_STATUS_W_NOT_BF16) == 0
    np.testing.assert_array_equal(a.codes(), b.codes())


@pytest.mark.parametrize("case,kw", [("ragged", {}), ("gqa8-b4", dict(center_query=True))])
def test_decode_step_against_the_oracle(mp, case, kw):
    wl = STEP_CASES[case]
    steps = [0, 15, 16, 17, 39] if case == "ragged" else [0, 11]
    rep = check_workload(mp, wl, WL.generate(wl), steps=steps, check_csr_tables=wl.L, use_step=True, **kw)
    _report(f"decode step {case}", rep)
