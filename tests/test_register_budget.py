"""The hot kernels compile for sm_103a without register spills (CPU only:
ptxas's resource report, `nvcc -Xptxas -v`, of the library's own sources).

Held to zero spill stores and loads:
- every instantiation of the table builder;
- the dp4a correlation's 128 x 32-tile family (four CTAs per SM at 64
  registers), which includes the 4096 x 4096 / 16 x 16 kernel;
- the bank kernel in pair mode (one exact group, at most 64 templates);
- every instantiation of the Toeplitz tensor-core kernel and of the
  transform kernels.
The dp4a kernel's 128 x 64-tile instantiations (three CTAs per SM) are not
held to it: under their register cap some spill a few hundred bytes.
"""
import concurrent.futures as cf
import os
import re
import shutil
import subprocess

import pytest

from normalized_cross_correlation_gb300 import _build

CSRC = os.path.join(os.path.dirname(_build.__file__), "csrc")
FILES = ["sat_build.cu", "correlate_dp4a.cu", "correlate_bank_tc.cu", "correlate_toeplitz_tc.cu",
         "correlate_ntt.cu"]
# (pattern on the mangled entry name, instantiations expected at least)
HOT = [
    (r"sat_build_kernelI", 7),
    (r"corr_dp4a_kernelI(?:Lb\dE){4}Li\d+ELb0ELi4E", 6),
    (r"bank_tc_kernelILb\dELb1ELb1E", 2),
    (r"toeplitz_tc_kernelI", 6),
    (r"ntt_corr_kernelI", 2),
    (r"ntt_spectrum_kernel", 1),
]


@pytest.fixture(scope="module")
def resource_report(tmp_path_factory):
    nvcc = shutil.which("nvcc") or os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    out = tmp_path_factory.mktemp("ptxas")

    def one(name):
        cmd = [nvcc, *_build.ARCH, *_build.CFLAGS, "-Xptxas", "-v", "-c", os.path.join(CSRC, name),
               "-o", str(out / (name + ".o"))]
        res = subprocess.run(cmd, capture_output=True, text=True)
        assert res.returncode == 0, res.stderr[-3000:]
        return res.stderr

    with cf.ThreadPoolExecutor(max_workers=len(FILES)) as ex:
        logs = list(ex.map(one, FILES))
    report = {}
    for log in logs:
        entry = None
        for line in log.splitlines():
            m = re.search(r"Compiling entry function '(\S+)'", line)
            if m:
                entry = m.group(1)
                continue
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and entry:
                report[entry] = (int(m.group(1)), int(m.group(2)))
                entry = None
    return report


@pytest.mark.parametrize("pattern,at_least", HOT)
def test_hot_kernels_do_not_spill(resource_report, pattern, at_least):
    hits = {name: s for name, s in resource_report.items() if re.search(pattern, name)}
    assert len(hits) >= at_least, sorted(resource_report)
    spilling = {name: s for name, s in hits.items() if s != (0, 0)}
    assert not spilling, spilling
