"""Mutation tests of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of oracle/q4q_oracle.c (a
dropped term, a wrong sign, index or divisor, a different rounding rule, the
absolute value taken in the wrong place), builds that copy, and runs the pin
files against it in a child process: at least one pin must fail.  A control
case runs the same harness on an unchanged copy, which must pass.

The mistakes are planted in the oracle, on the CPU, and nowhere else.  The
method is "llama.cpp 深度解读" (luoboask.github.io) §2 (the Q4_0 encode and
decode) and §3 (the block dot product), and the rows next to the matmul that
tests/test_oracle_pins_next.py pins (row gather, bias / GELU, SwiGLU, Q8_0
weights).
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "q4q_oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py"), os.path.join(ROOT, "tests", "test_oracle_pins_next.py")]

# name -> list of (text in q4q_oracle.c, replacement); every text must occur exactly once
MUTATIONS = {
    # Q4_0 encode (§2 steps 2-4)
    "q4_divisor_7": [("float scale = amax / 8.0f;", "float scale = amax / 7.0f;")],
    "q4_round_half_even": [("float r = roundf(w[k] / scale);        /* half away from zero */",
                            "float r = rintf(w[k] / scale);")],
    "q4_clamp_at_8": [("if (r > 7.0f) r = 7.0f;", "if (r > 8.0f) r = 8.0f;")],
    "q4_nibbles_swapped": [("out[2 + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));",
                            "out[2 + j] = (uint8_t)(q[2 * j + 1] | (q[2 * j] << 4));")],
    # Q8_0 encode
    "q8_divisor_128": [("float scale = amax / 127.0f;", "float scale = amax / 128.0f;")],
    "q8_round_half_even": [("float r = roundf(x[k] / scale);", "float r = rintf(x[k] / scale);")],
    # fp16 narrowing: ties go up instead of to even
    "fp16_ties_up": [("if (rem > half || (rem == half && (h & 1u))) h += 1u;", "if (rem >= half) h += 1u;")],
    # §3 block dot
    "dot_no_offset_low": [("int32_t v0 = (int32_t)(qs[j] & 0x0F) - 8;", "int32_t v0 = (int32_t)(qs[j] & 0x0F);")],
    "dot_activations_swapped": [("sumi += v0 * (int32_t)y[2 * j + 0] + v1 * (int32_t)y[2 * j + 1];",
                                 "sumi += v0 * (int32_t)y[2 * j + 1] + v1 * (int32_t)y[2 * j + 0];")],
    "dot_scale_drops_d1": [("float d = d0 * d1;", "float d = d0;")],
    "mul_mat_output_transposed": [("dst[i11 * ne01 + i01] = orc_vec_dot_q4_0_q8_0(ne00, xrow, yrow);",
                                   "dst[i01 * ne11 + i11] = orc_vec_dot_q4_0_q8_0(ne00, xrow, yrow);")],
    # the tolerance scale: |sum| instead of sum of |terms|
    "scale_abs_of_sum": [("        s += fabs((double)d * (double)block_isum(xb, yb));\n    }\n    return s;",
                          "        s += (double)d * (double)block_isum(xb, yb);\n    }\n    return fabs(s);")],
    "w8_scale_abs_of_sum": [("        s += fabs((double)d * (double)block_isum_w8(xb, yb));\n    }\n    return s;",
                             "        s += (double)d * (double)block_isum_w8(xb, yb);\n    }\n    return fabs(s);")],
    # rows next to the matmul
    "w8_codes_unsigned": [("for (int k = 0; k < ORC_QK; ++k) sumi += (int32_t)x[k] * (int32_t)y[k];",
                           "for (int k = 0; k < ORC_QK; ++k) sumi += (int32_t)(uint8_t)x[k] * (int32_t)y[k];")],
    "get_rows_off_by_one": [("int64_t id = ids[i];", "int64_t id = ids[i] + 1;")],
    "gelu_tanh_form": [("return 0.5 * x * erfc(-x / sqrt(2.0));",
                        "return 0.5 * x * (1.0 + tanh(0.7978845608028654 * (x + 0.044715 * x * x * x)));")],
    "silu_sign": [("return x * (1.0 / (1.0 + exp(-x)));", "return x * (1.0 / (1.0 + exp(x)));")],
    "bias_by_token": [("if (bias) v = v + bias[r];", "if (bias) v = v + bias[t];")],
    "swiglu_operands_swapped": [("float s = (float)orc_silu((double)gate[i]);\n        y[i] = s * up[i];",
                                 "float s = (float)orc_silu((double)up[i]);\n        y[i] = s * gate[i];")],
}


def _mutant_source(name):
    text = open(SRC, encoding="utf-8").read()
    for old, new in MUTATIONS.get(name, []):
        assert text.count(old) == 1, "mutation %s: the oracle text it targets changed" % name
        text = text.replace(old, new)
    return text


def _run_pins(name, workdir):
    d = os.path.join(workdir, name)
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, "q4q_oracle.c")
    with open(src, "w", encoding="utf-8") as f:
        f.write(_mutant_source(name))
    env = dict(os.environ, Q4Q_ORACLE_SRC=src, PYTHONDONTWRITEBYTECODE="1", OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                        "-W", "ignore::RuntimeWarning"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-3000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    work = str(tmp_path_factory.mktemp("oracle_mutants"))
    names = ["control"] + sorted(MUTATIONS)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        return dict(zip(names, ex.map(lambda n: _run_pins(n, work), names)))


def test_control_copy_passes_every_pin(outcomes):
    rc, log = outcomes["control"]
    assert rc == 0, log


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(outcomes, name):
    rc, log = outcomes[name]
    # exit code 1: tests ran and at least one failed (not a collection or build error)
    assert rc == 1, "mutation %s survived every pin (rc %d):\n%s" % (name, rc, log)
