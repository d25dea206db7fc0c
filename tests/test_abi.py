"""The C-ABI library builds, loads without a GPU and exports every entry
point include/*.h declares; argument checks answer before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                  if f.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ncc_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("ncc_sat_build", "ncc_correlate", "ncc_correlate_bank", "ncc_sync_status",
                 "ncc_status_string", "ncc_correlate_moments", "ncc_match", "ncc_match_host"):
        assert want in names


def test_library_exports_every_declared_symbol(built_lib):
    L = ctypes.CDLL(built_lib)
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in ncc.h but not exported"


def test_binding_lists_every_declared_symbol():
    from normalized_cross_correlation_gb300 import ncc
    assert sorted(ncc.EXPORTS) == declared_functions()


def test_status_strings_and_version(built_lib):
    from normalized_cross_correlation_gb300 import ncc
    assert ncc.ncc_status_string(0) == "ok"
    assert "time" in ncc.ncc_status_string(ncc.NCC_ERR_TIMEOUT)
    assert ncc.ncc_status_string(12345) == "unknown status"
    assert ncc.ncc_version() >= 1


def test_argument_checks_need_no_gpu(built_lib):
    from normalized_cross_correlation_gb300 import ncc
    L = ncc.lib()
    fake = 4096  # never dereferenced: every call below fails its checks first
    # null / non-positive sizes
    assert L.ncc_sat_build(None, 16, 16, fake, fake * 4, None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_sat_build(fake, 0, 16, fake * 4, fake * 8, None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_sat_build(fake, 16, -1, fake * 4, fake * 8, None) == ncc.NCC_ERR_INVALID_ARG
    # a row's running sum of squares must fit uint32: W <= 66051
    assert L.ncc_sat_build(fake, 66052, 1, fake * 4, fake * 8, None) == ncc.NCC_ERR_UNSUPPORTED
    # misaligned table pointers
    assert L.ncc_sat_build(fake, 16, 16, fake * 4 + 4, fake * 8, None) == ncc.NCC_ERR_INVALID_ARG
    # overlapping tables
    assert L.ncc_sat_build(fake, 16, 16, fake * 4, fake * 4 + 8, None) == ncc.NCC_ERR_INVALID_ARG
    # template larger than the image, empty bank
    assert L.ncc_correlate(fake, 16, 16, fake, 17, 4, fake * 8, fake * 16, fake * 32,
                           None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_correlate_bank(fake, 16, 16, fake, 4, 4, 0, fake * 8, fake * 16, fake * 32,
                                None) == ncc.NCC_ERR_INVALID_ARG
    # SumIT must fit uint32: wT*hT <= 66051
    assert L.ncc_correlate(fake, 300, 300, fake, 300, 300, fake * 1024, fake * 2048, fake * 4096,
                           None) == ncc.NCC_ERR_UNSUPPORTED
    # output overlapping an input
    assert L.ncc_correlate(fake, 16, 16, fake * 2, 4, 4, fake * 8, fake * 16, fake * 8,
                           None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_match_host(None, 16, 16, fake, 4, 4, 1, fake, None) == ncc.NCC_ERR_INVALID_ARG
    # the direct-moment calls: wider than 129 is refused, missing image, output over the image
    assert L.ncc_correlate_direct(fake, 200, 40, fake * 16, 130, 4, 1, fake * 32,
                                  None) == ncc.NCC_ERR_UNSUPPORTED
    assert L.ncc_correlate_direct(None, 200, 40, fake * 16, 16, 4, 1, fake * 32,
                                  None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_correlate_direct(fake, 200, 40, fake * 16, 16, 4, 1, fake + 64,
                                  None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_correlate_direct_moments(fake, 200, 40, fake * 16, 16, 4, 1, fake * 32,
                                          fake * 32 + 8, fake * 64, None) == ncc.NCC_ERR_INVALID_ARG
    # the combined call: missing image, overlapping tables, a table over the templates
    assert L.ncc_match(None, 16, 16, fake * 2, 4, 4, 1, fake * 8, fake * 16, fake * 32,
                       None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_match(fake, 16, 16, fake * 2, 4, 4, 1, fake * 8, fake * 8 + 8, fake * 32,
                       None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_match(fake, 16, 16, fake * 8 + 16, 4, 4, 1, fake * 8, fake * 16, fake * 32,
                       None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_match(fake, 16, 16, fake * 2, 4, 4, 1, fake * 8, fake * 16, fake * 8 + 64,
                       None) == ncc.NCC_ERR_INVALID_ARG
    # the no-alloc builder's fixed scratch holds at most 2729 tiles of 128x128:
    # 42 x 65 = 2730 tiles is refused before any device work
    assert L.ncc_sat_build_noalloc(fake, 128 * 42, 128 * 65, 1 << 32, (1 << 32) + (1 << 30),
                                   None) == ncc.NCC_ERR_UNSUPPORTED
    # the compared SAT builders: unknown variant, then the same checks as ncc_sat_build
    assert L.ncc_sat_build_variant(fake, 16, 16, fake * 4, fake * 8, 9, None) == ncc.NCC_ERR_INVALID_ARG
    for v in (ncc.NCC_SAT_FUSED, ncc.NCC_SAT_NAIVE, ncc.NCC_SAT_TWO_PASS):
        assert L.ncc_sat_build_variant(fake, 0, 16, fake * 4, fake * 8, v, None) == ncc.NCC_ERR_INVALID_ARG
        assert L.ncc_sat_build_variant(fake, 66052, 1, fake * 4, fake * 8, v, None) == ncc.NCC_ERR_UNSUPPORTED
        assert L.ncc_sat_build_variant(fake, 16, 16, fake * 4, fake * 4 + 8, v, None) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_debug_set_fault(-2, 0) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_debug_fail_alloc(-1) == ncc.NCC_ERR_INVALID_ARG
    assert L.ncc_debug_fail_alloc(0) == ncc.NCC_OK


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "normalized_cross_correlation_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f), errors="ignore").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "ncc_oracle" not in text, f


def test_binding_refuses_cpu_tensors():
    """The device entry points take CUDA tensors only: CPU tensors raise
    before any call, so nothing is ever computed on the host."""
    import torch
    from normalized_cross_correlation_gb300 import ncc
    img = torch.zeros((64, 64), dtype=torch.uint8)
    T = torch.zeros((8, 8), dtype=torch.uint8)
    S = torch.zeros((64, 64), dtype=torch.int64)
    calls = [
        lambda: ncc.ncc_sat_build(img),
        lambda: ncc.ncc_sat_build_variant(img, ncc.NCC_SAT_NAIVE),
        lambda: ncc.ncc_correlate(img, T, S, S),
        lambda: ncc.ncc_correlate_bank(img, T[None], S, S),
        lambda: ncc.ncc_correlate_moments(img, T, S, S),
        lambda: ncc.ncc_correlate_direct(img, T),
        lambda: ncc.ncc_correlate_direct_moments(img, T),
        lambda: ncc.ncc_match(img, T),
    ]
    for call in calls:
        with pytest.raises(TypeError):
            call()


def test_host_entry_point_checks_dtypes_and_output_shape(monkeypatch):
    """ncc_match_host refuses host buffers of the wrong dtype, layout or
    output shape before it calls the library."""
    import numpy as np
    from normalized_cross_correlation_gb300 import ncc

    def refuse():
        raise AssertionError("the binding reached the library with bad arguments")
    monkeypatch.setattr(ncc, "lib", refuse)
    img = np.zeros((64, 80), np.uint8)
    T = np.zeros((1, 8, 6), np.uint8)
    refused = [
        lambda: ncc.ncc_match_host(img.astype(np.int16), T),
        lambda: ncc.ncc_match_host(img, T.astype(np.float32)),
        lambda: ncc.ncc_match_host(img, T, out=np.zeros((1, 57, 74), np.float32)),
        lambda: ncc.ncc_match_host(img, T, out=np.zeros((1, 57, 75), np.float64)),
        lambda: ncc.ncc_match_host(img[:, ::2], T),
    ]
    for call in refused:
        with pytest.raises((TypeError, ValueError)):
            call()


def test_header_is_plain_c_and_links(built_lib, tmp_path):
    """include/ncc.h and ncc_debug.h compile as strict C99 (no C++ or CUDA headers needed),
    and a C program links against the library and calls it without a GPU."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "use_ncc.c"
    src.write_text(
        '#include "ncc.h"\n'
        '#include "ncc_debug.h"\n'
        "int main(void) {\n"
        "    if (ncc_version() <= 0) return 1;\n"
        "    if (ncc_sat_build(0, 16, 16, 0, 0, 0) != NCC_ERR_INVALID_ARG) return 2;\n"
        "    return ncc_status_string(NCC_OK)[0] == 'o' ? 0 : 3;\n"
        "}\n")
    exe = tmp_path / "use_ncc"
    libdir = os.path.dirname(built_lib)
    name = os.path.basename(built_lib)[3:-3]          # libX.so -> X
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-l" + name,
                    "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    assert subprocess.run([str(exe)]).returncode == 0
