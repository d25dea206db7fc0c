"""The debug build of the library (libncc_gb300_debug.so, compiled with
NCC_DEBUG): every kernel checks its hand-computed indices -- shared-memory
offsets, tensor-memory columns, the ranges of its MMA operand descriptors,
table rows and output addresses -- and reports a failed check as
NCC_ERR_BOUNDS through the status word, skipping the access (no trap).

1. The small-shape parity suites pass against the debug build: every GPU test
   there ends with ncc_sync_status() == NCC_OK, so no check failed on any of
   their shapes (ragged tiles, unaligned rows, every kernel and path).
2. A planted out-of-range store (the debug build's ncc_debug_set_fault(-2)
   hook moves tile 0's table stores one row width to the left, before the
   start of the tables) is caught:
   the status reads NCC_ERR_BOUNDS, nothing faults, and the next build is
   exact."""
import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUITES = ["tests/test_sat_gpu.py", "tests/test_correlate_gpu.py",
          "tests/test_correlate_toeplitz_gpu.py", "tests/test_correlate_ntt_gpu.py",
          "tests/test_bank_gpu.py",
          "tests/test_direct_gpu.py", "tests/test_match_gpu.py",
          "tests/test_sat_ladder_gpu.py"]

PLANTED = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, {root!r})
import oracle
from normalized_cross_correlation_gb300 import ncc
assert ncc.library_path().endswith("_debug.so"), ncc.library_path()
img_np = np.random.default_rng(31).integers(0, 256, (300, 500), dtype=np.uint8)
img = torch.from_numpy(img_np).cuda()
ncc.ncc_debug_set_fault(-2, 0)         # tile 0's stores go one row width to the left
try:
    ncc.ncc_sat_build(img)
    status = ncc.ncc_sync_status()
finally:
    ncc.ncc_debug_set_fault(-1, 0)
if status != ncc.NCC_ERR_BOUNDS:
    sys.exit(10)
S, Q = ncc.ncc_sat_build(img)           # normal again, and exact
if ncc.ncc_sync_status() != ncc.NCC_OK:
    sys.exit(11)
oS, oQ = oracle.sat(img_np)
sys.exit(0 if np.array_equal(S.cpu().numpy(), oS) and np.array_equal(Q.cpu().numpy(), oQ) else 12)
"""


@pytest.fixture(scope="module")
def debug_env(ncc):
    from normalized_cross_correlation_gb300 import _build
    _build.build(debug=True)
    env = dict(os.environ)
    env["NCC_GB300_LIBRARY"] = "debug"
    return env


def test_small_parity_suites_pass_on_the_debug_build(debug_env):
    cmd = [sys.executable, "-m", "pytest", *SUITES, "-m", "gpu", "-q", "-x",
           "-k", "not 4096 and not 8192 and not headline"]
    res = subprocess.run(cmd, cwd=ROOT, env=debug_env, capture_output=True, text=True, timeout=1500)
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-2000:]
    m = re.search(r"(\d+) passed", res.stdout)
    assert m and int(m.group(1)) >= 100, res.stdout[-2000:]   # the suites really ran


def test_planted_out_of_range_store_is_caught(debug_env):
    res = subprocess.run([sys.executable, "-c", PLANTED.format(root=ROOT)], cwd=ROOT, env=debug_env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, (res.returncode, res.stdout[-2000:], res.stderr[-2000:])


def test_regular_build_refuses_the_planting_hook(ncc):
    with pytest.raises(ncc.NccError) as e:
        ncc.ncc_debug_set_fault(-2, 0)
    assert e.value.code == ncc.NCC_ERR_INVALID_ARG
