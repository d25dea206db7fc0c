"""Rate probes behind the rooflines of the correlation kernels.

    python -m normalized_cross_correlation_gb300.peaks [--compile-only]

Builds each probe in this folder for sm_103a with nvcc into a temporary
directory and runs it on GPU 0:

* ``dp4a_rate.cu``    -- dp4a / IMAD / PRMT+IADD operations per SM per clock;
* ``tcgen05_rate.cu`` -- tcgen05.mma kind::f16 rates for the operand layouts
  of the bank and Toeplitz kernels, with and without barrier hand-offs;
* ``i8_assembles.cu`` -- assembled (never run) for sm_103a and sm_100a, to
  report which target accepts the integer tcgen05.mma.

``--compile-only`` builds everything and runs nothing (no GPU needed).
"""
import argparse
import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
NVCC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")


def nvcc(src, out, arch="103a", extra=()):
    cmd = [NVCC, "-O3", "-std=c++17", f"-gencode=arch=compute_{arch},code=sm_{arch}",
           *extra, "-o", out, os.path.join(HERE, src)]
    return subprocess.run(cmd, capture_output=True, text=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--compile-only", action="store_true")
    args = ap.parse_args(argv)
    rc = 0
    with tempfile.TemporaryDirectory() as tmp:
        for arch in ("103a", "100a"):
            r = nvcc("i8_assembles.cu", os.path.join(tmp, f"i8_{arch}.o"), arch, ("-c",))
            errs = [ln for ln in r.stderr.splitlines() if "error" in ln.lower()] or ["?"]
            msg = "accepted" if r.returncode == 0 else "rejected: " + errs[0].split("error", 1)[-1].strip(" :")
            print(f"kind::i8 tcgen05.mma on sm_{arch}: {msg}")
        for src in ("dp4a_rate.cu", "tcgen05_rate.cu"):
            exe = os.path.join(tmp, src[:-3])
            r = nvcc(src, exe)
            if r.returncode != 0:
                print(r.stderr, file=sys.stderr)
                return 1
            if args.compile_only:
                print(f"built {src}")
                continue
            print(f"--- {src}")
            run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
            print(run.stdout, end="")
            flags = [tok for tok in run.stdout.split() if tok.startswith("err=")]
            if run.returncode != 0 or any(f != "err=0" for f in flags):
                print(run.stderr, file=sys.stderr)
                rc = run.returncode or 1
    return rc


if __name__ == "__main__":
    sys.exit(main())
