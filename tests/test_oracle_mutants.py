"""The pins have teeth: each test plants one plausible mistake in a copy of
the oracle (on the CPU), builds it, and runs the pin suite against it; at
least one pin must fail.  An unmodified copy must pass, so the failures come
from the planted mistakes."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

ORACLE_C = os.path.join(ROOT, "oracle", "oracle.c")
ORACLE_H = os.path.join(ROOT, "oracle", "oracle.h")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("average divides by N+1", "a[i] = a[i] / (float)N;", "a[i] = a[i] / (float)(N + 1);"),
    ("fp32 average multiplies by RN(1/N)", "a[i] = a[i] / (float)N;",
     "a[i] = a[i] * (1.0f / (float)N);"),
    # (the same mistake in the per-hop bf16 branch is not one: for every bf16
    # sum and every N up to 64 both quotients round to the same bf16)
    ("fp32-accumulating average multiplies by RN(1/N)",
     "a[i] = orc_bf16_to_f32(orc_f32_to_bf16(a[i] / (float)N));",
     "a[i] = orc_bf16_to_f32(orc_f32_to_bf16(a[i] * (1.0f / (float)N)));"),
    ("sum instead of average", "a[i] = a[i] / (float)N;\n            } else if (R->dt == ORC_BF16_ACC32)",
     "a[i] = a[i];\n            } else if (R->dt == ORC_BF16_ACC32)"),
    ("bf16 rounds half up", "b += 0x7fffu + ((b >> 16) & 1u);", "b += 0x8000u;"),
    ("bf16 truncates", "b += 0x7fffu + ((b >> 16) & 1u);", "b += 0u;"),
    ("reduce-scatter sends the wrong chunk", "ch[r] = pmod((int64_t)r - t - rho, N);",
     "ch[r] = pmod((int64_t)r + t - rho, N);"),
    ("all-gather starts from chunk r", "ch[r] = pmod((int64_t)r + 1 - rho - t, N);",
     "ch[r] = pmod((int64_t)r - rho - t, N);"),
    ("owner off by one", "return (int)pmod((int64_t)c - 1 + rho, N);",
     "return (int)pmod((int64_t)c + rho, N);"),
    ("bytes counted twice", "            if (sent) sent[r] += (int64_t)bytes;\n        }\n        /* then every",
     "            if (sent) sent[r] += 2 * (int64_t)bytes;\n        }\n        /* then every"),
    ("no weight decay", "theta[i] = th - lr * (upd + wd * th);", "theta[i] = th - lr * upd;"),
    ("weight decay not scaled by lr", "theta[i] = th - lr * (upd + wd * th);",
     "theta[i] = th - (lr * upd + wd * th);"),
    ("beta1 and beta2 swapped", "float mi = b1 * m[i] + omb1 * g;", "float mi = b2 * m[i] + omb2 * g;"),
    ("no bias correction of m", "float mhat = mi / bc1;", "float mhat = mi;"),
    ("eps inside the square root", "float upd = mhat / (sqrtf(vhat) + eps);",
     "float upd = mhat / sqrtf(vhat + eps);"),
    ("v from g instead of g*g", "float vi = b2 * v[i] + omb2 * (g * g);",
     "float vi = b2 * v[i] + omb2 * g;"),
    ("clip compares the wrong way", "if (clip > 0.0f && n > clip) s = clip / n;",
     "if (clip > 0.0f && n < clip) s = clip / n;"),
    ("norm sums |g|", "            double g = load_as_double(R->dt, p, i);\n            ss += g * g;",
     "            double g = load_as_double(R->dt, p, i);\n            ss += fabs(g);"),
    ("bias correction with beta1 for v", "*bc2 = (float)(1.0 - pow((double)cfg->beta2, (double)cfg->step));",
     "*bc2 = (float)(1.0 - pow((double)cfg->beta1, (double)cfg->step));"),
    ("fp32-accumulating ring rounds every hop",
     "    } else if (dt == ORC_F32 || dt == ORC_BF16_ACC32) {\n        float* a = (float*)local;\n        const float* b = (const float*)msg;\n        for (int64_t i = 0; i < n; ++i) a[i] = a[i] + b[i];",
     "    } else if (dt == ORC_F32 || dt == ORC_BF16_ACC32) {\n        float* a = (float*)local;\n        const float* b = (const float*)msg;\n        for (int64_t i = 0; i < n; ++i) a[i] = dt == ORC_F32 ? a[i] + b[i] : orc_bf16_to_f32(orc_f32_to_bf16(a[i] + b[i]));"),
]


def _build(tmp_path, text):
    src = tmp_path / "oracle.c"
    src.write_text(text)
    (tmp_path / "oracle.h").write_text(open(ORACLE_H).read())
    so = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", str(src), "-o", str(so), "-lm"])
    return str(so)


def _run_pins(so):
    env = dict(os.environ, DPZ_ORACLE_LIB=so)
    return subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                          capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)


def test_unmodified_copy_passes(tmp_path):
    out = _run_pins(_build(tmp_path, open(ORACLE_C).read()))
    assert out.returncode == 0, out.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(ORACLE_C).read()
    assert text.count(old) == 1, f"mutation site for {name!r} not unique"
    out = _run_pins(_build(tmp_path, text.replace(old, new)))
    assert out.returncode != 0, f"no pin caught: {name}"
