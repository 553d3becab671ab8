"""The oracle's pins catch plausible mistakes: each mutant below plants one
(a dropped term, a wrong sign, offset, bias or index, transposed operands, a
missing or wrong rounding) in a copy of the oracle's C source, builds it with
the oracle's own flags, and runs the pin tests against it (through
SGQ_ORACLE_LIBRARY); at least one pin must fail. The unmutated source, built
and run the same way, must pass them all. Runs on the CPU."""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

from oracle.build import SRC, compile_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(ROOT, "_build", "oracle_mutants")
PINS = ["tests/test_oracle_codecs.py", "tests/test_oracle_norm.py", "tests/test_oracle_swiglu.py",
        "tests/test_oracle_fp16.py", "tests/test_oracle_allreduce.py", "tests/test_oracle_layouts.py",
        "tests/test_oracle_flags.py"]

# (name, text in the oracle source, its replacement)
MUTANTS = [
    ("residual_dropped", "h[j] = io_decode(f16, xi[j]) + (r ? io_decode(f16, r[i * H + j]) : 0.0);",
     "h[j] = io_decode(f16, xi[j]);"),
    ("eps_dropped", "double inv = 1.0 / sqrt(ss / (double)H + (double)eps);",
     "double inv = 1.0 / sqrt(ss / (double)H + 0.0 * (double)eps);"),
    ("sum_not_mean", "double inv = 1.0 / sqrt(ss / (double)H + (double)eps);", "double inv = 1.0 / sqrt(ss + (double)eps);"),
    ("gemma_weight_swapped", "((flags & ORA_F_GEMMA) ? 1.0 + wj : wj)", "((flags & ORA_F_GEMMA) ? wj : 1.0 + wj)"),
    ("gemma_weight_sign", "((flags & ORA_F_GEMMA) ? 1.0 + wj : wj)", "((flags & ORA_F_GEMMA) ? 1.0 - wj : wj)"),
    ("bf16_truncates", "double n = nearbyint(a / ulp);", "double n = floor(a / ulp);"),
    ("e4m3_ties_to_odd", "(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)"),
    ("e4m3_bias", "else mag = (1.0 + m / 8.0) * ldexp(1.0, e - 7);", "else mag = (1.0 + m / 8.0) * ldexp(1.0, e - 6);"),
    ("mx_offset", "int e = (e2 - 1) - 8;", "int e = (e2 - 1) - 7;"),
    ("mx_scaling_sign", "double tj = src[j] * ldexp(1.0, -e);", "double tj = src[j] * ldexp(1.0, e);"),
    ("fp8_divisor", "float s = (float)(amax / 448.0);", "float s = (float)(amax / 447.0);"),
    ("amax_ignores_sign", "if (fabs(src[j]) > amax) amax = fabs(src[j]);", "if (src[j] > amax) amax = src[j];"),
    ("per_token_group", "return fmt == ORA_MXFP8 ? 32 : fmt == ORA_BLOCK128 ? 128 : width;",
     "return fmt == ORA_MXFP8 ? 32 : fmt == ORA_BLOCK128 ? 128 : width / 2;"),
    ("gate_up_transposed", "double g = ora_bf16_decode(row[j]), u = ora_bf16_decode(row[I + j]);",
     "double u = ora_bf16_decode(row[j]), g = ora_bf16_decode(row[I + j]);"),
    ("gate_clamped_below", "double gc = fmin(g, (double)limit);", "double gc = fmax(fmin(g, (double)limit), -(double)limit);"),
    ("beta_sign", "a[j] = gc * sigmoid((double)alpha * gc) * (uc + (double)beta);",
     "a[j] = gc * sigmoid((double)alpha * gc) * (uc - (double)beta);"),
    ("sigmoid_sign", "static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }",
     "static double sigmoid(double z) { return 1.0 / (1.0 + exp(z)); }"),
    ("silu_not_rounded", "s = ora_bf16_decode(ora_bf16_round(s));", "(void)0;"),
    ("source_never_rounded", "src[j] = from_fp32 ? pre[j] : io_decode(f16, io_round(f16, pre[j]));", "src[j] = pre[j];"),
    ("fp16_bias", "else v = ldexp(1024.0 + (double)f, e - 25);", "else v = ldexp(1024.0 + (double)f, e - 24);"),
    ("allreduce_last_rank", "for (int r = 0; r < n; ++r) s += io_decode(f16, parts[r][j]);",
     "for (int r = 0; r < n; ++r) s = io_decode(f16, parts[r][j]);"),
    # the ambiguity flags the parity checker relies on
    ("pow2_flag_always", "    if (amax == 0.0) return 0;\n    int e2;\n    double f = frexp(amax, &e2);     /* f in [0.5, 1) */",
     "    if (amax == 0.0) return 0;\n    if (rel > 0.0) return 1;\n    int e2;\n    double f = frexp(amax, &e2);     /* f in [0.5, 1) */"),
    ("tie_window_wide", "near_e4m3_boundary(tj, ldexp(1.0, -22))", "near_e4m3_boundary(tj, ldexp(1.0, -12))"),
    ("source_flag_dropped", "src_amb[j] = (unsigned char)(from_fp32 ? 0 : near_io_boundary(f16, pre[j], rel));",
     "src_amb[j] = (unsigned char)(0 * near_io_boundary(f16, pre[j], rel));"),
]


def _run_pins(name: str, text: str) -> tuple:
    """Build the oracle from `text` and run the pins against it; (pytest's
    exit code, the first failing pin or "")."""
    src = os.path.join(OUT, name + ".c")
    with open(src, "w") as f:
        f.write(text)
    so = compile_oracle(src, os.path.join(OUT, name + ".so"))
    env = dict(os.environ, SGQ_ORACLE_LIBRARY=so)
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT,
                       env=env, capture_output=True, text=True)
    failed = [ln.split()[1] for ln in r.stdout.splitlines() if ln.startswith("FAILED ")]
    return r.returncode, failed[0] if failed else ""


@pytest.fixture(scope="module")
def outcomes():
    os.makedirs(OUT, exist_ok=True)
    with open(SRC) as f:
        base = f.read()
    jobs = {"unmutated": base}
    for name, old, new in MUTANTS:
        assert base.count(old) == 1, f"{name}: the text to mutate must occur exactly once"
        jobs[name] = base.replace(old, new)
    with cf.ThreadPoolExecutor(max(1, min(8, (os.cpu_count() or 2) // 2))) as ex:
        codes = dict(zip(jobs, ex.map(lambda kv: _run_pins(*kv), jobs.items())))
    return codes


def test_unmutated_oracle_passes_the_pins(outcomes):
    assert outcomes["unmutated"] == (0, "")


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_fails_a_pin(outcomes, name):
    # exit code 1: tests ran and at least one failed (not a collection or usage error)
    code, pin = outcomes[name]
    assert code == 1 and pin, f"mutant {name}: pytest exit code {code}"
    print(f"{name}: caught by {pin}")
