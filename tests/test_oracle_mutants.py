"""Mistakes planted in copies of the oracle must each fail at least one pin.

Each mutant is wq_oracle.c with one plausible slip (a swapped index, a wrong
sign, a dropped term, a transposed operand, a wrong exponent bias...).  It is
compiled to a temporary library and the full pin suite runs against it in a
child process; the child exits 0 only if every pin passed, which would mean
the pins cannot see that mistake.  Everything here runs on the CPU.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "wq_oracle.c")

MUTANTS = {
    "weight-row-col-swap": ("field(qw[(size_t)(k / pack) * N + n], k % pack, w_bit);\n            double z",
                            "field(qw[(size_t)(k % pack) * N + n], k / pack, w_bit);\n            double z"),
    "zero-sign": ("wrow[j] = (q - z) * s;", "wrow[j] = (q + z) * s;"),
    "scale-column": ("double s = decode16(scales[(size_t)g * N + n], s_is_bf16);\n            wrow",
                     "double s = decode16(scales[(size_t)g * N], s_is_bf16);\n            wrow"),
    "x-transposed": ("double xv = decode16(x[(size_t)m * K + k], x_is_bf16);",
                     "double xv = decode16(x[(size_t)k * M + m], x_is_bf16);"),
    "zero-slot": ("field(qzeros[(size_t)(g / pack) * N + n], g % pack, w_bit)",
                  "field(qzeros[(size_t)(g / pack) * N + n], g / pack, w_bit)"),
    "shift-not-scaled": ("(word >> (slot * w_bit)) & mask", "(word >> slot) & mask"),
    "int8-q-transposed": ("(double)q[(size_t)n * K + k]", "(double)q[(size_t)k * N + n]"),
    "f16-bias": ("e - 25);     /* (1 + f/2^10)", "e - 24);     /* (1 + f/2^10)"),
    "bf16-hidden-bit": ("(128 + f), e - 134)", "(127 + f), e - 134)"),
    "dropped-accumulate": ("yr[j] += xv * wrow[j];", "yr[j] = xv * wrow[j];"),
    "symmetric-zero": ("return (double)(1 << (w_bit - 1));", "return (double)(1 << w_bit);"),
    "int8-scale-index": ("wq_oracle_f32_to_f64(scale_bits[n]) * acc", "wq_oracle_f32_to_f64(scale_bits[0]) * acc"),
    "group-index": ("int g = k / group_size;\n        /* row k", "int g = (k / group_size) / 2;\n        /* row k"),
    "dequant-zero-sign": ("w[(size_t)k * N + n] = (q - z) * s;", "w[(size_t)k * N + n] = (q + z) * s;"),
    "t2-plane-row-swap": ("(packed[(size_t)(k % R) * N + n] >> (2 * (k / R)))",
                          "(packed[(size_t)(k / R) * N + n] >> (2 * (k % R)))"),
    "t2-no-offset": ("& 3u) - 1;\n}", "& 3u);\n}"),
    "t2-field-width": ("(packed[(size_t)(k % R) * N + n] >> (2 * (k / R))) & 3u)",
                       "(packed[(size_t)(k % R) * N + n] >> (k / R)) & 3u)"),
    "dequant-scale-row": ("double s = decode16(scales[(size_t)g * N + n], s_is_bf16);\n            w[",
                          "double s = decode16(scales[(size_t)(k % (K / group_size)) * N + n], s_is_bf16);\n            w["),
}

CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import oracle_pins
orc = oracle.load({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(orc)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED_PINS", failed)
sys.exit(1 if failed else 0)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site not found: " + name
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                           "-o", str(lib), str(mut), "-lm"])
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, lib=str(lib))],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, "mutant %s passed every pin:\n%s%s" % (name, r.stdout, r.stderr)
