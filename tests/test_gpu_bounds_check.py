"""The bounds-checking build (MP_CHECK=1) over the small GPU parity cases.

compute-sanitizer is not available to these tests, so the library has a build in which
every kernel index that comes from data (codes, bucket offsets, list entries) is tested
against its buffer before use; a failure sets MP_STATUS_BAD_INDEX in the status word and
skips the access. The parity harness asserts a clear status word after every call, so
running the parity cases on that build checks that no such index ever leaves its buffer.
The cases run in a child process, which loads libmagicpig_check.so (MP_BOUNDS_CHECK=1)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    ("tests/test_gpu_parity.py",
     "config0 or config1 or ragged or thresholds or K0 or short or tile_layouts or scan_match_mode "
     "or decode_step or dtypes or centering_off or status_flags"),
    ("tests/test_gpu_geometry.py", "constant_key or center_query_both or tight_cone_layer"),
]


def test_parity_cases_on_the_bounds_checking_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MP_BOUNDS_CHECK="1")
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_mp_build", os.path.join(ROOT, "lsh_sampled_sparse_centered_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build(check=True)
    for path, sel in CASES:
        r = subprocess.run([sys.executable, "-m", "pytest", path, "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
                            "-k", sel], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
        assert r.returncode == 0, (path, r.stdout[-3000:], r.stderr[-2000:])
        assert " passed" in r.stdout, r.stdout[-500:]
