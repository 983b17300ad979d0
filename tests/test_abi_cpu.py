"""C-ABI checks that need no GPU: the library loads, exports every declared
entry point, validates arguments and injects faults on the host before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "magicpig.h")


@pytest.fixture(scope="module")
def mp():
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as m
    return m


def _declared():
    src = open(HEADER).read()
    return re.findall(r"MP_API\s+[\w\s\*]+?\b(mp_\w+)\s*\(", src)


def test_every_declared_symbol_is_exported(mp):
    names = _declared()
    assert len(names) >= 9
    out = subprocess.run(["nm", "-D", "--defined-only", mp.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s+(mp_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(mp.LIB_PATH)
    for n in names:
        assert getattr(lib, n) is not None
    assert set(mp.EXPORTED) <= set(names)
    assert mp.mp_abi_version() == 4


def _cfg(mp, **kw):
    base = dict(layers=1, batch=1, kv_heads=2, q_heads=4, head_dim=128, K=8, L=75, n_sink=4, window=64,
                capacity=4096, dtype="bf16")
    base.update(kw)
    return mp.make_config(**base)


def test_config_validation(mp):
    assert mp.mp_config_check(_cfg(mp)) == mp.MP_OK
    assert mp.mp_config_check(_cfg(mp, threshold=3)) == mp.MP_OK
    assert mp.mp_config_check(_cfg(mp, threshold=7, capacity=200000, match_mode=2)) == mp.MP_OK
    bad = [dict(q_heads=3), dict(layers=0), dict(K=-1), dict(L=0), dict(capacity=0), dict(dtype=7),
           dict(threshold=0), dict(window=-1), dict(match_mode=9)]
    for b in bad:
        assert mp.mp_config_check(_cfg(mp, **b)) == mp.MP_ERR_INVALID_ARG, b
    unsup = [dict(head_dim=96), dict(K=13), dict(L=2000), dict(capacity=(1 << 19) + 1), dict(threshold=8),
             dict(threshold=3, L=300), dict(threshold=3, capacity=200000, match_mode=1)]
    for u in unsup:
        assert mp.mp_config_check(_cfg(mp, **u)) == mp.MP_ERR_UNSUPPORTED, u
    c = _cfg(mp)
    c.reserved[1] = 1
    assert mp.mp_config_check(c) == mp.MP_ERR_INVALID_ARG
    assert mp.mp_config_check(_cfg(mp, centering=False)) == mp.MP_OK
    c = _cfg(mp)
    c.no_centering = 2
    assert mp.mp_config_check(c) == mp.MP_ERR_INVALID_ARG
    # both query readings are accepted, with and without key centering
    assert mp.mp_config_check(_cfg(mp, center_query=True)) == mp.MP_OK
    assert mp.mp_config_check(_cfg(mp, center_query=True, centering=False)) == mp.MP_OK
    c = _cfg(mp)
    c.center_query = 2
    assert mp.mp_config_check(c) == mp.MP_ERR_INVALID_ARG


def test_layouts_are_aligned_disjoint_and_sized(mp):
    c = _cfg(mp, layers=2, w_per_layer=True)
    t = mp.mp_tables_layout_get(c)
    names = ["header", "center", "beta", "ones", "negbeta_f32", "wt_f32", "wt_bf16", "center_parts", "codes", "csr_offsets",
             "csr_ids", "logu_lut"]
    offs = [getattr(t, n) for n in names]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs) and len(set(offs)) == len(offs)
    U, L, cap, d = 2 * 1 * 2, 75, 4096, 128
    assert t.csr_offsets - t.codes >= U * L * cap * 2
    assert t.logu_lut - t.csr_ids >= U * L * cap * 2
    assert t.total_bytes - t.logu_lut >= (4096 + 1) * 4                # -log u on the cosine grid
    assert t.tc_cols == 768 and t.n_buckets == 256
    assert t.wt_bf16 - t.wt_f32 >= 2 * 768 * d * 4
    assert t.center_parts - t.wt_bf16 >= 2 * 3 * 768 * d * 2      # hi, mid, lo bf16 terms of W
    assert t.wt_f32 - t.negbeta_f32 >= U * 768 * 4                  # fp32 -beta per unit and column
    assert t.negbeta_f32 - t.ones >= 128 * 16 * 2
    assert t.ones - t.beta >= U * 768 * 16 * 2
    ns = -(-cap // 32768)
    assert t.csr_ids - t.csr_offsets >= U * L * (256 + 1) * ns * 2  # bucket-major offsets
    dl = mp.mp_decode_layout_get(c)
    Q = 2 * 4
    assert dl.lists % 256 == 0 and dl.partials - dl.lists >= Q * cap * 4
    assert dl.total_bytes - dl.counters >= (Q + 1) * 4            # + the attention's work queue
    f32 = mp.mp_tables_layout_get(_cfg(mp, dtype="f32"))
    assert f32.wt_bf16 == 0


def test_argument_errors_return_before_any_launch(mp):
    c = _cfg(mp)
    fake = 1 << 20  # never dereferenced: validation fails first
    assert mp.call_raw("mp_build_tables", ctypes.byref(c), None, 10, fake, fake, None) == mp.MP_ERR_INVALID_ARG
    assert mp.call_raw("mp_build_tables", ctypes.byref(c), fake, 0, fake, fake, None) == mp.MP_ERR_CAPACITY
    assert mp.call_raw("mp_build_tables", ctypes.byref(c), fake, 5000, fake, fake, None) == mp.MP_ERR_CAPACITY
    assert mp.call_raw("mp_build_tables", ctypes.byref(c), fake + 8, 10, fake, fake, None) == mp.MP_ERR_INVALID_ARG
    assert mp.call_raw("mp_append", ctypes.byref(c), fake, fake, 4096, None) == mp.MP_ERR_CAPACITY
    assert mp.call_raw("mp_append", ctypes.byref(c), fake, fake, -1, None) == mp.MP_ERR_CAPACITY
    dl = mp.mp_decode_layout_get(c)
    assert mp.call_raw("mp_decode_attention", ctypes.byref(c), fake, fake, fake, 100, fake, fake, fake,
                       ctypes.c_size_t(dl.total_bytes - 1), None) == mp.MP_ERR_SCRATCH
    assert mp.call_raw("mp_decode_attention", ctypes.byref(c), fake, fake, fake, 0, fake, fake, fake,
                       ctypes.c_size_t(dl.total_bytes), None) == mp.MP_ERR_CAPACITY
    assert mp.call_raw("mp_decode_attention", ctypes.byref(c), fake, fake, None, 100, fake, fake, fake,
                       ctypes.c_size_t(dl.total_bytes), None) == mp.MP_ERR_INVALID_ARG
    # the decode step: the appended position bounds the capacity, the scratch size as above
    assert mp.call_raw("mp_decode_step", ctypes.byref(c), fake, fake, fake, 4096, fake, fake, fake,
                       ctypes.c_size_t(dl.total_bytes), None) == mp.MP_ERR_CAPACITY
    assert mp.call_raw("mp_decode_step", ctypes.byref(c), fake, fake, fake, -1, fake, fake, fake,
                       ctypes.c_size_t(dl.total_bytes), None) == mp.MP_ERR_CAPACITY
    assert mp.call_raw("mp_decode_step", ctypes.byref(c), fake, fake, fake, 100, fake, fake, fake,
                       ctypes.c_size_t(dl.total_bytes - 1), None) == mp.MP_ERR_SCRATCH
    assert mp.call_raw("mp_decode_step", ctypes.byref(c), fake, fake, fake, 100, fake, None, fake,
                       ctypes.c_size_t(dl.total_bytes), None) == mp.MP_ERR_INVALID_ARG
    assert mp.call_raw("mp_get_status", None, None, None) == mp.MP_ERR_INVALID_ARG
    assert mp.mp_status_string(mp.MP_ERR_SCRATCH) == "scratch buffer too small"


def test_fault_injection_on_the_host(mp, monkeypatch):
    c = _cfg(mp)
    fake = 1 << 20
    dl = mp.mp_decode_layout_get(c)
    monkeypatch.setenv("MP_FAULT_INJECT", "decode")
    assert mp.call_raw("mp_decode_attention", ctypes.byref(c), fake, fake, fake, 100, fake, fake, fake,
                       ctypes.c_size_t(dl.total_bytes), None) == mp.MP_ERR_INJECTED
    monkeypatch.setenv("MP_FAULT_INJECT", "all")
    assert mp.call_raw("mp_build_tables", ctypes.byref(c), fake, 10, fake, fake, None) == mp.MP_ERR_INJECTED
    assert mp.call_raw("mp_append", ctypes.byref(c), fake, fake, 20, None) == mp.MP_ERR_INJECTED
    assert mp.call_raw("mp_decode_step", ctypes.byref(c), fake, fake, fake, 100, fake, fake, fake,
                       ctypes.c_size_t(dl.total_bytes), None) == mp.MP_ERR_INJECTED
    with pytest.raises(mp.MagicPigError) as e:
        mp.mp_append(c, fake, fake, 20, stream=0)
    assert e.value.code == mp.MP_ERR_INJECTED


def test_binding_refuses_host_and_strided_tensors(mp):
    import pytest
    import torch
    c = _cfg(mp)
    host = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(ValueError):
        mp.mp_build_tables(c, host, 10, host, host, stream=0)
    with pytest.raises(ValueError):
        mp._ptr(torch.zeros(4, 4)[:, 1])


def test_auto_match_mode_picks_the_fewer_bytes(mp):
    """AUTO compares bytes per query head: the bucket walk reads L·m/2^K ids plus the
    ranges; the bit-plane scan reads m·L·K/8 bytes shared by the G query heads of a
    KV head. Long contexts with 4-head groups (the bench shape) walk buckets; a short
    context with large groups and K = 1 streams the planes."""
    big = _cfg(mp, kv_heads=8, q_heads=32, K=10, L=150, capacity=98368)
    assert mp.mp_tables_layout_get(big).match_mode == mp.MP_MATCH_CSR
    small = _cfg(mp, kv_heads=1, q_heads=64, K=1, L=8, capacity=2048)
    assert mp.mp_tables_layout_get(small).match_mode == mp.MP_MATCH_SCAN
    forced = _cfg(mp, kv_heads=1, q_heads=64, K=1, L=8, capacity=2048, match_mode=mp.MP_MATCH_CSR)
    assert mp.mp_tables_layout_get(forced).match_mode == mp.MP_MATCH_CSR


def test_bounds_checking_build_exports_the_same_entry_points(mp):
    """The MP_CHECK=1 library (built on request) declares and exports what the ordinary one
    does, and refuses the same bad arguments before any launch."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_mp_build", os.path.join(os.path.dirname(mp.__file__), "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    path = b.build(check=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s+(mp_\w+)", out))
    assert set(_declared()) <= exported
    lib = ctypes.CDLL(path)
    c = _cfg(mp)
    lib.mp_config_check.argtypes = [ctypes.POINTER(mp.mp_config)]
    assert lib.mp_config_check(ctypes.byref(c)) == mp.MP_OK
    c.K = 13
    assert lib.mp_config_check(ctypes.byref(c)) == mp.MP_ERR_UNSUPPORTED
