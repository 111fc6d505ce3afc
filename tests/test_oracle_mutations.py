"""The oracle's pins catch plausible mistakes in it.

Each case copies oracle/oracle.c, plants one mistake (a swapped GQA map, an
off-by-one causal offset, a dropped scale or normaliser, a wrong row inside
a block, a wrong write slot, an off-by-one window start, a wrong E4M3
exponent bias, rounding, saturation or scale), compiles the copy
with the same gcc flags and runs tests/test_oracle_pins.py against it: the
pins must fail.  The unmodified copy, built the same way, must pass.  The
mistakes are planted in the CPU oracle only; nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, replacement, occurrences)
MUTATIONS = [
    ("gqa_interleaved", "int32_t kh = h / g;", "int32_t kh = h % P->hkv;", 1),
    ("causal_offset", "int64_t p = (int64_t)L - t + i;", "int64_t p = (int64_t)L - t + i - 1;", 1),
    ("scale_dropped", "s *= P->scale;", "s *= 1.0;", 1),
    ("normaliser_dropped", "out_row[e] /= l;", "out_row[e] /= 1.0;", 1),
    ("row_in_block", "int64_t slot = (int64_t)blk * P->bs + j % P->bs;",
     "int64_t slot = (int64_t)blk * P->bs + (j + 1) % P->bs;", 2),
    ("write_slot", "return (int64_t)table_row[p / bs] * bs + p % bs;",
     "return (int64_t)table_row[p / bs] * bs + (bs - 1 - p % bs);", 1),
    ("window_start", "j0 = p - P->window + 1;", "j0 = p - P->window;", 1),
    ("e4m3_bias", "v = (1.0 + man / 8.0) * ldexp(1.0, field - 7);",
     "v = (1.0 + man / 8.0) * ldexp(1.0, field - 8);", 1),
    ("round_half_up", "if (r > 0.5 || (r == 0.5 && fmod(f, 2.0) != 0.0))", "if (r >= 0.5)", 1),
    ("saturate_to_nan", "return sign | 0x7E;", "return sign | 0x7F;", 1),
    ("fp8_scale_max", "float scale = amax / 448.0f;", "float scale = amax / 240.0f;", 1),
]


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(src),
                           "-lm"])
    return str(lib)


def _run_pins(lib):
    env = dict(os.environ, PKV_ORACLE_LIB=lib, OMP_NUM_THREADS="4")
    return subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                           "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


def test_unmodified_copy_passes(tmp_path):
    r = _run_pins(_build(tmp_path, "same", open(SRC).read()))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_the_pins(tmp_path, name, old, new, count):
    text = open(SRC).read()
    assert text.count(old) == count, f"{name}: the oracle no longer contains {old!r}"
    r = _run_pins(_build(tmp_path, name, text.replace(old, new)))
    assert r.returncode != 0 and "failed" in r.stdout, f"{name} was not caught:\n{r.stdout[-2000:]}"
