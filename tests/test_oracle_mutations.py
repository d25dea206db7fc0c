"""Plants plausible mistakes in a copy of the oracle's C source (on the CPU
only), builds each copy, and checks that the pin tests reject every one.
This shows that the pins would catch a dropped term, a wrong sign, a shifted
or transposed index, or a wrong zero-variance rule in the oracle itself."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ncc_oracle.c")

MUTATIONS = {
    "sat_drops_row_above": ("S[at(W, x, y)] = above_i + run_i;", "S[at(W, x, y)] = run_i;"),
    "sat_q_not_squared": ("run_q += p * p;", "run_q += p;"),
    "box_wrong_sign": ("+ table_at(S, W, x0 - 1, y0 - 1);", "- table_at(S, W, x0 - 1, y0 - 1);"),
    "box_off_by_one": ("return table_at(S, W, x1 - 1, y1 - 1)", "return table_at(S, W, x1, y1 - 1)"),
    "template_transposed": ("T[at(wT, dx, dy)]", "T[at(hT, dy, dx)]"),
    "window_square_uses_template": ("s2 += p * p;", "s2 += p * t;"),
    "num_wrong_sign": ("int64_t num = N * sIT - sI * sT;", "int64_t num = N * sIT + sI * sT;"),
    "vI_wrong_term": ("int64_t vI = N * sI2 - sI * sI;", "int64_t vI = N * sI2 - sI * sT;"),
    "zero_variance_rule_dropped": ("if (vI == 0 || vT == 0) return 0.0;", "if (vT == 0) return 0.0;"),
    "image_row_stride_wrong": ("img[at(W, x + dx, y + dy)]", "img[at(W - 1, x + dx, y + dy)]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutated.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutated.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", str(mutated), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, NCC_ORACLE_LIB=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"pins did not catch mutation {name}:\n{res.stdout[-2000:]}"
