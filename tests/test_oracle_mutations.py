"""The oracle's pins catch plausible mistakes in it.

Each case plants one mistake in a copy of oracle/ftoracle.c (a wrong exponent bias, a tie broken the wrong way, a
dropped term, a swapped operand, a wrong index), builds it with the oracle's own flags, and runs the oracle pin
suites against it (FT_ORACLE_LIB points the oracle's Python wrapper at the altered library).  Every altered oracle
must fail at least one pin.  CPU only; nothing here touches a GPU or the CUDA library.
"""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ftoracle.c")
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_quant.py", "tests/test_oracle_route_permute.py",
        "tests/test_oracle_ffn.py"]

# (name, text in ftoracle.c, replacement)
MUTATIONS = [
    ("e2m1 exponent bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    ("e4m3 exponent bias", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    ("e4m3 subnormal step", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    ("e2m1 ties to odd", "c = (i % 2 == 0) ? i : i + 1;", "c = (i % 2 == 0) ? i + 1 : i;"),
    ("e2m1 sign inverted", "((v < 0.0f) ? 8 : 0)", "((v > 0.0f) ? 8 : 0)"),
    ("e4m3 ties down", "return (uint8_t)((lo % 2 == 0) ? lo : lo + 1);", "return (uint8_t)lo;"),
    ("bf16 with 9 significant bits", "? e - 8 : -133", "? e - 9 : -133"),
    ("block scale amax/4", "const float d = amax / 6.0f;", "const float d = amax / 4.0f;"),
    ("tensor scale amax/448", "float st = amax / 2688.0f;", "float st = amax / 448.0f;"),
    ("nibbles swapped", "packed[j] = (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));",
     "packed[j] = (uint8_t)((codes[2 * j] << 4) | codes[2 * j + 1]);"),
    ("tensor scale dropped in dequantisation", "ora_e2m1_value(c) * s * tensor_scale;", "ora_e2m1_value(c) * s;"),
    ("router ties to the higher index", "if (best < 0 || l[e] > l[best]) best = e;",
     "if (best < 0 || l[e] >= l[best]) best = e;"),
    ("router weights not renormalised", "for (int j = 0; j < k; ++j) den += exp((double)l[ids[(int64_t)t * k + j]] - m);",
     "for (int e = 0; e < E; ++e) den += exp((double)l[e] - m);"),
    ("permutation not stable", "const int32_t p = offsets[e] + fill[e]++;",
     "const int32_t p = offsets[e + 1] - 1 - fill[e]++;"),
    ("silu dropped", "h[i] = ora_bf16_round(silu(g) * u);", "h[i] = ora_bf16_round(g * u);"),
    ("gate and up swapped", "h[i] = ora_bf16_round(silu(g) * u);", "h[i] = ora_bf16_round(silu(u) * g);"),
    ("h not rounded to bf16", "h[i] = ora_bf16_round(silu(g) * u);", "h[i] = silu(g) * u;"),
    ("down projection rows reversed", "y[r * H + n] = dot(Wd + n * I, h, I);",
     "y[r * H + n] = dot(Wd + (H - 1 - n) * I, h, I);"),
    ("combine weights in reverse slot order", "s += w[(int64_t)t * k + j] * y",
     "s += w[(int64_t)t * k + (k - 1 - j)] * y"),
    ("combined output not rounded", "out[(int64_t)t * H + n] = ora_bf16_round(s);", "out[(int64_t)t * H + n] = s;"),
    ("A4 mode skips the x quantisation", "deq_vec(qc, qs, H, xa);", "memcpy(xa, xr, sizeof(double) * (size_t)H);"),
    ("negative zero kept", "if (c == 0) return 0;", "if (c == 0 && v >= 0.0f) return 0;"),
    ("zero tensor keeps a zero scale", "if (st == 0.0f) st = 1.0f;", "if (st < 0.0f) st = 1.0f;"),
    ("all -inf row weighted 0", "for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = 1.0 / k;",
     "for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = 0.0;"),
    ("offsets not shifted", "for (int64_t f = 0; f < n; ++f) offsets[ids[f] + 1] += 1;",
     "for (int64_t f = 0; f < n; ++f) offsets[ids[f] + (ids[f] + 1 < E)] += 1;"),
    ("combine ignores inv", "y[(int64_t)inv[(int64_t)t * k + j] * H + n]", "y[((int64_t)t * k + j) * H + n]"),
    ("e4m3 NaN code read as a number", "if ((b & 0x7F) == 0x7F) return NAN;", "if (b == 0xFF) return NAN;"),
    ("bf16 overflow kept finite", "if (fabs(r) >= 0x1.0p128) return v > 0 ? INFINITY : -INFINITY;",
     "if (fabs(r) >= 0x1.0p129) return v > 0 ? INFINITY : -INFINITY;"),
    ("e2m1 saturates to 4", "    int c = 7;\n    if (a < 6.0) {", "    int c = 6;\n    if (a < 6.0) {"),
]


def run_pins_on_mutant(tmp, idx, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    c_path = os.path.join(tmp, f"m{idx}.c")
    so_path = os.path.join(tmp, f"m{idx}.so")
    with open(c_path, "w") as fh:
        fh.write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
                           "-shared", "-o", so_path, c_path, "-lm"])
    env = dict(os.environ, FT_ORACLE_LIB=so_path, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-1500:]


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            futs = {name: ex.submit(run_pins_on_mutant, tmp, i, old, new)
                    for i, (name, old, new) in enumerate(MUTATIONS)}
            results = {name: f.result() for name, f in futs.items()}
    survived = [name for name, (rc, _) in results.items() if rc == 0]
    assert not survived, f"mistakes no pin caught: {survived}"
    # a failure must be a pin failing, not the test run breaking
    broken = [name for name, (rc, out) in results.items() if rc not in (0, 1)]
    assert not broken, {name: results[name][1] for name in broken}
