"""Strength of the oracle's pins: plant one plausible mistake at a time in a copy of oracle.c and
check that tests/test_oracle.py fails on it (and passes on an unmodified copy).

Each mistake is one that would otherwise survive: a wrong offset, sign, index, nibble or byte order,
a dropped term, a different rounding or tie rule.  The copies live in oracle/_mutants/ (not tracked).
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
OUT = os.path.join(ROOT, "oracle", "_mutants")

# (name, original text, planted mistake); every original text occurs in oracle.c
MUTATIONS = [
    ("q4_0_offset", "if (type == ORC_Q4_0) return code - 8;", "if (type == ORC_Q4_0) return code - 7;"),
    ("tile_nibble_order", "tile[cp * 32 + r] = (uint8_t)(((c1 & 0x0F) << 4) | (c0 & 0x0F));",
     "tile[cp * 32 + r] = (uint8_t)(((c0 & 0x0F) << 4) | (c1 & 0x0F));"),
    ("q8_tile_interleave", "tile[cp * 64 + 2 * r + 0] = (uint8_t)(int8_t)c0;", "tile[cp * 64 + 2 * r + 1] = (uint8_t)(int8_t)c0;"),
    ("tile_index", "return ct * n_k_tiles + kt; }", "return kt * n_k_tiles + ct; }"),
    ("q4k_high_bits", "*sc = (scales[j + 4] & 0x0F) | ((scales[j - 4] >> 6) << 4);",
     "*sc = (scales[j + 4] & 0x0F) | ((scales[j] >> 6) << 4);"),
    ("q4k_min_sign", "orc_f32_to_f16(-(dmin * (float)m))", "orc_f32_to_f16(dmin * (float)m)"),
    ("q4k_nibble", "return (sb[16 + 32 * (j / 2) + i] >> (4 * (j & 1))) & 15;",
     "return (sb[16 + 32 * (j / 2) + i] >> (4 * ((j + 1) & 1))) & 15;"),
    ("q4k_scale_rounding", "sc[j] = clamp63(scale[j] * isc + 0.5f);", "sc[j] = clamp63(scale[j] * isc);"),
    ("q4_1_min_dropped", "acc += dw * da * (double)s + mw * da * (double)asum;", "acc += dw * da * (double)s;"),
    ("q4_1_rounding", "float v = (x[j] - mn) * id + 0.5f;", "float v = (x[j] - mn) * id + 0.49f;"),
    ("act_half_to_even", "else r = roundf(v);", "else r = rintf(v);"),
    ("act_x_over_d", "float v = x[j] * id;\n        float r;", "float v = x[j] / d;\n        float r;"),
    ("q4_0_tie_last", "if (fabsf(x[j]) > amax) { amax = fabsf(x[j]); m = x[j]; }",
     "if (fabsf(x[j]) >= amax) { amax = fabsf(x[j]); m = x[j]; }"),
    ("q4_0_d_sign", "float d = m / -8.0f;", "float d = m / 8.0f;"),
    ("table_ties_highest", "if (err < best_err) { best_err = err; best = i; }", "if (err <= best_err) { best_err = err; best = i; }"),
    ("mxfp4_exponent", "e = (ex - 1) - 2 + 127;", "e = (ex - 1) - 1 + 127;"),
    ("mxfp4_scale_bias", "int f = e - 112;", "int f = e - 111;"),
    ("f16_ties", "if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) n = fl + 1.0;", "if (rem >= 0.5) n = fl + 1.0;"),
    ("bound_abs", "sabs += (w * a < 0) ? -(w * a) : (w * a);", "sabs += w * a;"),
]


def _run_pins(name, text):
    os.makedirs(OUT, exist_ok=True)
    path = os.path.join(OUT, f"{name}.c")
    with open(path, "w") as f:
        f.write(text)
    env = dict(os.environ, QMM_ORACLE_SRC=path)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_unmodified_copy_passes():
    assert _run_pins("unmodified", open(SRC).read()) == 0


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    src = open(SRC).read()
    assert old in src, "the original text moved; update the mutation"
    assert _run_pins(name, src.replace(old, new)) != 0, f"the pins did not catch: {name}"
