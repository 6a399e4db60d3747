"""The pins are strong enough: each plausible mistake planted in a copy of
the oracle (a dropped term, a wrong sign or index, a transposed operand, an
off-by-one mask) makes the pin suite fail.  The mutants are compiled from
the oracle source into a temporary directory; the real oracle is untouched."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fa_oracle.c")

MUTANTS = {
    "dQ without scale": ("acc += dS[(int64_t)i * N + j] * Kh[(int64_t)j * d + t];\n                    dQh[(int64_t)i * d + t] = scale * acc;",
                         "acc += dS[(int64_t)i * N + j] * Kh[(int64_t)j * d + t];\n                    dQh[(int64_t)i * d + t] = acc;"),
    "rect dQ without scale": ("acc += dS[(int64_t)i * Nk + j] * Kh[(int64_t)j * d + t];\n                dQh[(int64_t)i * d + t] = scale * acc;",
                              "acc += dS[(int64_t)i * Nk + j] * Kh[(int64_t)j * d + t];\n                dQh[(int64_t)i * d + t] = acc;"),
    "dK transposed dS": ("ak += dS[(int64_t)i * N + j] * Qh[(int64_t)i * d + t];",
                         "ak += dS[(int64_t)j * N + i] * Qh[(int64_t)i * d + t];"),
    "dS sign of D": ("dS[(int64_t)i * N + j] = p * (dp - Dv[i]);", "dS[(int64_t)i * N + j] = p * (dp + Dv[i]);"),
    "dV from dS": ("av += P[(int64_t)i * N + j] * dOh[(int64_t)i * d + t];",
                   "av += dS[(int64_t)i * N + j] * dOh[(int64_t)i * d + t];"),
    "causal off by one": ("if (causal && j > i) return 0;", "if (causal && j >= i) return 0;"),
    "key_len off by one": ("if (key_len && j >= key_len[b]) return 0;", "if (key_len && j > key_len[b]) return 0;"),
    "block mask transposed": ("block_mask[(int64_t)(i / mask_block) * nb + j / mask_block]",
                              "block_mask[(int64_t)(j / mask_block) * nb + i / mask_block]"),
    "softmax not normalised": ("for (int j = 0; j < N; j++) s[j] = exp(s[j] - m) / l;",
                               "for (int j = 0; j < N; j++) s[j] = exp(s[j] - m);"),
    "LSE drops the max": ("return m + log(l);", "return log(l);"),
    "score without scale": ("        for (int t = 0; t < d; t++) acc += q[t] * k[t];\n        s[j] = scale * acc;",
                            "        for (int t = 0; t < d; t++) acc += q[t] * k[t];\n        s[j] = acc;"),
    "decode score without scale": ("acc += q[t] * Kh[(int64_t)j * d + t];\n            s[j] = scale * acc;",
                                   "acc += q[t] * Kh[(int64_t)j * d + t];\n            s[j] = acc;"),
    "decode causal offset": ("if (causal && j > len - Nq + i) vis = 0;", "if (causal && j > len - Nq + i + 1) vis = 0;"),
    "decode kv_len off by one": ("int vis = j < len;", "int vis = j <= len;"),
    "e4m3 ties away from even": ("(frac == 0.5 && fmod(r, 2.0) != 0.0)", "(frac == 0.5)"),
    "e4m3 exponent bias 8": ("const int field = (E2 - 1) + 7;", "const int field = (E2 - 1) + 8;"),
    "fp8 scale for a 240 maximum": ("amax > 0.0f ? amax / 448.0f : 0.0f", "amax > 0.0f ? amax / 240.0f : 0.0f"),
    "fp8 transposed row stride": ("codes[(bh * d + c) * Np + r] = code;", "codes[(bh * d + c) * N + r] = code;"),
    "rect backward causal top-left": ("if (causal && j > i + (Nk - Nq)) {", "if (causal && j > i) {"),
    "rect dV from dS": ("av += P[(int64_t)i * Nk + j] * dOh[(int64_t)i * d + t];",
                        "av += dS[(int64_t)i * Nk + j] * dOh[(int64_t)i * d + t];"),
    "rect dK without scale": ("dKh[(int64_t)j * d + t] = scale * ak;\n                dVh[(int64_t)j * d + t] = av;\n            }\n    }",
                              "dKh[(int64_t)j * d + t] = ak;\n                dVh[(int64_t)j * d + t] = av;\n            }\n    }"),
    "D without dO": ("acc += dOh[(int64_t)i * d + t] * Oh[(int64_t)i * d + t];",
                     "acc += Oh[(int64_t)i * d + t];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(mut), "-lm"],
                   check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_fp8_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant '%s' survived the pins" % name
