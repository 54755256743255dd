"""The pins must reject a broken oracle.

Each case plants one plausible mistake in a temporary copy of the oracle's C
source (on the CPU; the real oracle is untouched), builds it, and runs the pin
suite against it through FP8Q_ORACLE_LIB.  A mutation that every pin accepts
would mean the pins do not constrain that part of the definition.
"""
import os
import subprocess
import sys
import tempfile

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "fp8q_oracle.c")

# (name, original text, planted replacement)
MUTATIONS = [
    ("ties away instead of to even (fp8)", "else code = (lo % 2 == 0) ? lo : hi;", "else code = hi;"),
    ("no saturation", "return (uint8_t)(sign | maxc);", "return 0x7F;"),
    ("multiply by the reciprocal instead of dividing", "float y = x / scale;", "float y = x * (1.0f / scale);"),
    ("amax without abs", "m = amax_combine(m, fabsf(x));", "m = amax_combine(m, x);"),
    ("roll toward newer", "hist[(int64_t)h * S + s] = hist[(int64_t)(h - 1) * S + s];",
     "hist[(int64_t)(h - 1) * S + s] = hist[(int64_t)h * S + s];"),
    ("margin sign", "sc = ldexpf(sc, margin);", "sc = ldexpf(sc, -margin);"),
    ("dequantize divides", "float p = v * scale;", "float p = v / scale;"),
    ("bf16 ties away", "else pick = ((lo >> 16) & 1u) ? hi : lo;", "else pick = hi;"),
    ("selection algos swapped", "if (algo == ORC_ALGO_MAX)", "if (algo != ORC_ALGO_MAX)"),
    ("subnormal exponent off by one", "v = ldexp((double)m, 1 - bias - mbits);", "v = ldexp((double)m, - bias - mbits);"),
    ("scale inverted", "float sc = a / fp8max;", "float sc = fp8max / a;"),
    ("scale_inv not inverted", "*scale_inv = 1.0f / sc;", "*scale_inv = sc;"),
    ("subnormal scale accepted", "if (!isnormal(sc)) return;", "if (!isfinite(sc)) return;"),
    ("dropped roll insert", "hist[s] = amax_new[s];", "(void)amax_new;"),
    ("ring overwrites the newest entry", "h = (h + 1) % H;", "h = h % H;"),
    ("ring window one row short", "for (int32_t r = 0; r < H; ++r) a = amax_combine(a, hist[(int64_t)r * S + s]);",
     "for (int32_t r = 0; r < H - 1; ++r) a = amax_combine(a, hist[(int64_t)r * S + s]);"),
    ("GELU cubic term dropped", "const double u = k * (x + 0.044715 * x * x * x);", "const double u = k * x;"),
    ("GELU exponent sign flipped", "return x / (1.0 + exp(-2.0 * u));", "return x / (1.0 + exp(2.0 * u));"),
    ("bf16 from float64 rounds through binary32 first", "double a = fabs(g);", "double a = fabs((double)(float)g);"),
    ("bf16 from float64 ties away", "else pick = (fmod(m, 2.0) == 0.0) ? lo : hi;", "else pick = hi;"),
    ("LayerNorm without beta", "* (rstd * (double)gamma[i]) + (double)beta[i];", "* (rstd * (double)gamma[i]);"),
    ("LayerNorm without gamma", "* (rstd * (double)gamma[i]) + (double)beta[i];", "* rstd + (double)beta[i];"),
    ("LayerNorm without eps", "double rstd = 1.0 / sqrt(var + eps);", "double rstd = 1.0 / sqrt(var);"),
    ("LayerNorm variance without the mean's square", "double var = s2 / H - mean * mean;", "double var = s2 / H;"),
    ("fused Q->DQ divides on the way back", "float p = (float)orc_fp8_decode(code, fmt) * scale;",
     "float p = (float)orc_fp8_decode(code, fmt) / scale;"),
]


def _build_mutant(tmp, i, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, old
    d = os.path.join(tmp, f"m{i}")
    os.makedirs(d)
    with open(os.path.join(d, "fp8q_oracle.c"), "w") as f:
        f.write(src.replace(old, new))
    with open(os.path.join(d, "fp8q_oracle.h"), "w") as f:
        f.write(open(os.path.join(ROOT, "oracle", "fp8q_oracle.h")).read())
    lib = os.path.join(d, "lib.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", lib,
                    os.path.join(d, "fp8q_oracle.c"), "-lm"], check=True)
    return lib


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        procs = []
        for i, (name, old, new) in enumerate(MUTATIONS):
            lib = _build_mutant(tmp, i, old, new)
            env = dict(os.environ, FP8Q_ORACLE_LIB=lib)
            p = subprocess.Popen([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                                  os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                                 cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
            procs.append((name, p))
        survivors = []
        for name, p in procs:
            out, _ = p.communicate(timeout=600)
            if p.returncode == 0:
                survivors.append(name)
        assert not survivors, f"pins accepted mutated oracles: {survivors}"
