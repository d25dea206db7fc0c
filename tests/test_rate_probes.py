"""The rate probes behind the rooflines build for sm_103a (CPU only: nvcc,
nothing runs), and the assembler's answer on the integer tensor-core MMA
that decides the bank kernel's operand type: tcgen05.mma kind::i8 is
rejected for sm_103a and accepted for sm_100a, so the bank multiplies u8
values converted exactly to f16 (kind::f16) instead."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_rate_probes_build_and_i8_mma_is_rejected_on_sm_103a():
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not found")
    res = subprocess.run([sys.executable, "-m", "normalized_cross_correlation_gb300.peaks",
                          "--compile-only"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = res.stdout.splitlines()
    assert any(l.startswith("kind::i8 tcgen05.mma on sm_103a: rejected") for l in lines), res.stdout
    assert "kind::i8 tcgen05.mma on sm_100a: accepted" in lines, res.stdout
    assert "built dp4a_rate.cu" in lines and "built tcgen05_rate.cu" in lines, res.stdout
