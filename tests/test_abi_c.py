"""The library from C: a C99 program that includes only `include/magicpig.h` and links
`libmagicpig.so` compiles warning-free, and the calls that need no GPU return the
documented codes. The struct sizes it prints must equal those of the Python binding's
ctypes mirrors, so that the header and the binding describe the same memory."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mp():
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as m
    return m


def test_c_caller_sees_the_documented_codes_and_sizes(mp, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(mp.LIB_PATH)
    exe = str(tmp_path / "abi_from_c")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "abi_from_c.c"), "-L", libdir, "-lmagicpig",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    assert int(got["abi"]) == 4
    assert int(got["sizeof_config"]) == ctypes.sizeof(mp.mp_config)
    assert int(got["sizeof_tables_layout"]) == ctypes.sizeof(mp.mp_tables_layout)
    assert int(got["sizeof_decode_layout"]) == ctypes.sizeof(mp.mp_decode_layout)
    assert int(got["sizeof_kernel_time"]) == ctypes.sizeof(mp.mp_kernel_time)
    assert int(got["check_ok"]) == mp.MP_OK
    assert int(got["check_null"]) == mp.MP_ERR_INVALID_ARG
    assert int(got["check_bad_group"]) == mp.MP_ERR_INVALID_ARG
    assert int(got["check_head_dim"]) == mp.MP_ERR_UNSUPPORTED
    assert int(got["tables_layout"]) == mp.MP_OK and int(got["decode_layout"]) == mp.MP_OK
    cfg = mp.make_config(layers=1, batch=1, kv_heads=2, q_heads=4, head_dim=128, K=8, L=75, n_sink=4,
                         window=64, capacity=4096, dtype="bf16")
    assert int(got["tables_bytes"]) == mp.mp_tables_layout_get(cfg).total_bytes
    assert int(got["tables_match_mode"]) == mp.mp_tables_layout_get(cfg).match_mode
    assert int(got["decode_bytes"]) == mp.mp_decode_layout_get(cfg).total_bytes
    assert int(got["build_capacity"]) == mp.MP_ERR_CAPACITY
    assert int(got["build_null_keys"]) == mp.MP_ERR_INVALID_ARG
    assert int(got["append_capacity"]) == mp.MP_ERR_CAPACITY
    assert int(got["decode_scratch"]) == mp.MP_ERR_SCRATCH
    assert got["status_string"] == mp.mp_status_string(mp.MP_ERR_CAPACITY)
