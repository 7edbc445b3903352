"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle source to a temporary directory, plants one
mistake (a dropped term, a wrong sign or index, a transposed operand, an
off-by-one), builds it, and runs the pin suite against that copy in a child
process.  The committed oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

MUTANTS = {
    "score_sign": ("x *= scale;", "x *= -scale;"),
    "no_max_shift_in_lse": ("double w = exp(work[j - lo] - m);", "double w = exp(work[j - lo]);"),
    "gqa_interleaved": ("int g = h / group;", "int g = h % kv_heads;"),
    "causal_top_left": ("int64_t p = kend - qlen + i;", "int64_t p = i;"),
    "window_off_by_one": ("last - window + 1 > 0) *lo = last - window + 1;",
                          "last - window > 0) *lo = last - window;"),
    "ring_not_wrapped": ("int64_t r = P->ring_rows ? pos % P->ring_rows : pos;", "int64_t r = pos;"),
    "page_offset_transposed": ("const double *kv = k_pool + ((b * ORACLE_BLOCK + off) * kv_heads + g) * D;",
                               "const double *kv = k_pool + ((off * ORACLE_BLOCK + b) * kv_heads + g) * D;"),
    "append_at_length": ("int64_t pos = (int64_t)seg[3] - seg[1] + i;", "int64_t pos = (int64_t)seg[3] + i;"),
    "no_normalisation": ("for (int d = 0; d < D; ++d) o[d] /= sum;", ""),
    "non_causal_masked": ("*hi = causal ? p + 1 : kend;", "*hi = p + 1;"),
    "tail_step_floor": ("int64_t steps = (over + kTailStep - 1) / kTailStep;",
                        "int64_t steps = over / kTailStep + 1;"),
    "v_from_k": ("const double *vv = v_pool +", "const double *vv = k_pool +"),
    "padding_keys_not_hidden": ("} else if (*lo < first) {", "} else if (0) {"),
    "padding_row_sees_prefix": ("*lo = p;\n", "*lo = 0;\n"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(lib), str(mut), "-lm"])
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
