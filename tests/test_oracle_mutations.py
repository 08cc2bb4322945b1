"""Planted mistakes: each mutation of the oracle's C source (one dropped
term, wrong sign, swapped index or operand) must make at least one pin fail.
The mutated oracles are built and run on the CPU in child processes."""

import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qmoe_oracle.c")

MUTATIONS = [
    ("nibble order", "uint8_t nib = (kk & 1) ? (byte >> 4) : (byte & 15);",
     "uint8_t nib = (kk & 1) ? (byte & 15) : (byte >> 4);"),
    ("int4 offset", "return (double)((int)(n & 15) - 8);", "return (double)((int)(n & 15) - 7);"),
    ("e2m1 exponent", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    ("e4m3 bias", "v = ldexp(8.0 + m, e - 10);", "v = ldexp(8.0 + m, e - 9);"),
    ("e8m0 bias", "ldexp(1.0, (int)b - 127)", "ldexp(1.0, (int)b - 126)"),
    ("silu sign", "return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    ("gate/up swapped", "dequant_row(scheme, (const uint8_t*)w1, w1s, 2 * I, H, e, I + n, wrow);",
     "dequant_row(scheme, (const uint8_t*)w1, w1s, 2 * I, H, e, n, wrow);"),
    ("mx emax", "int X = (ex - 1) - 8;", "int X = (ex - 1) - 7;"),
    ("routing weight dropped", "for (int c = 0; c < H; ++c) o[c] += wt * y[c];",
     "for (int c = 0; c < H; ++c) o[c] += y[c];"),
    ("w8a8 channel scale dropped", "float gf = ((float)ag * sa) * sw[n];", "float gf = ((float)ag * sa);"),
    ("int8 weights transposed", "memcpy(out, (const int8_t*)w + ((int64_t)e * R + row) * K, (size_t)K);",
     "memcpy(out, (const int8_t*)w + (int64_t)e * R * K + row, (size_t)K);"),
    ("w4a8 nibble order", "uint8_t code = (uint8_t)((wr[kk / 2] >> (4 * (kk % 2))) & 15);",
     "uint8_t code = (uint8_t)((wr[kk / 2] >> (4 - 4 * (kk % 2))) & 15);"),
    ("w4a8 gate/up swapped", "int_row(scheme, w1, 2 * I, H, e, I + n, wu);", "int_row(scheme, w1, 2 * I, H, e, n, wu);"),
    ("combine weight dropped",
     "for (int c = 0; c < H; ++c) out[t * H + c] += w * (double)y[(int64_t)s * H + c];",
     "for (int c = 0; c < H; ++c) out[t * H + c] += (double)y[(int64_t)s * H + c];"),
    ("combine unrouted pair read", "if (s < 0) continue;", "if (s < 0) s = 0;"),
    ("int8 rounding", "float t = rintf(vr[i] / sc);", "float t = truncf(vr[i] / sc);"),
    ("stable order", "int32_t s = cursor[e]++;", "int32_t s = offsets[e + 1] - 1 - (cursor[e]++ - offsets[e]);"),
    ("scale block index", "sc = oracle_e8m0_to_double(((const uint8_t*)ws)[sbase + kk / 32]);",
     "sc = oracle_e8m0_to_double(((const uint8_t*)ws)[sbase + kk / 64]);"),
]

PINS = ["tests/test_oracle_pins.py"]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {name}"
    mutated = tmp_path / "qmoe_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    str(mutated), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, QMOE_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation '{name}' survived every pin"
