"""The oracle's pins catch plausible mistakes: each mutant below plants one
mistake in a copy of ``oracle/fp8_oracle.c`` (a wrong bias, sign, rounding
rule, index or bound, a dropped or transposed term), and the oracle's pin files
(``test_oracle_e4m3.py``, ``test_oracle_quant.py``, ``test_oracle_gemm.py``)
run unchanged against that copy must fail. The unmutated copy must pass, so a
failure is the mistake's and not the harness's.

Every mutant keeps all accesses in bounds, so a pin that fails does so on a
value, never on a crash. The copies live in a temporary tree with their own
build folder; the committed oracle is not touched.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ["test_oracle_e4m3.py", "test_oracle_quant.py", "test_oracle_gemm.py", "test_oracle_rowwise.py",
             "test_oracle_kv_cache.py"]

# (name, snippet of fp8_oracle.c, replacement); each snippet occurs exactly once.
MUTANTS = [
    # E4M3 decode
    ("decode: bias 8", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("decode: no implicit leading one", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "mag = ldexp((double)m / 8.0, e - 7);"),
    ("decode: subnormal exponent -7", "mag = ldexp((double)m / 8.0, -6);", "mag = ldexp((double)m / 8.0, -7);"),
    ("decode: sign dropped", "return s ? -mag : mag;", "return mag;"),
    ("decode: 0x7E taken as NaN", "if (e == 15 && m == 7)", "if (e == 15 && m >= 6)"),
    # E4M3 encode
    ("encode: overflow to NaN instead of saturating", "return sign | 0x7E;", "return sign | 0x7F;"),
    ("encode: ties away from zero", "n = nearbyint(a / quantum);", "n = round(a / quantum);"),
    ("encode: truncation", "n = nearbyint(a / quantum);", "n = floor(a / quantum);"),
    ("encode: sign of zero dropped", "if (a == 0.0)\n        return sign;", "if (a == 0.0)\n        return 0;"),
    ("encode: subnormal spacing one binade too fine", "if (exponent < -6)\n        exponent = -6;",
     "if (exponent < -7)\n        exponent = -7;"),
    ("encode: two mantissa bits", "quantum = ldexp(1.0, exponent - 3);", "quantum = ldexp(1.0, exponent - 2);"),
    ("encode: subnormal code off by a factor 2", "return (uint8_t)(r / ldexp(1.0, -9));",
     "return (uint8_t)(r / ldexp(1.0, -8));"),
    ("encode: values that round above 448 give NaN", "if (a >= ORA_E4M3_MAX)\n        return sign | 0x7E;",
     "if (a >= 464.0)\n        return sign | 0x7F;\n    if (a >= ORA_E4M3_MAX)\n        return sign | 0x7E;"),
    ("bulk encoder: off by one pattern", "cv.u = first + (uint32_t)i;", "cv.u = first + (uint32_t)i + 1u;"),
    # scale and codes
    ("scale: no amax floor", "float a = amax > ORA_AMAX_FLOOR ? amax : ORA_AMAX_FLOOR;", "float a = amax;"),
    ("scale: divides by 480", "return (float)((double)a / ORA_E4M3_MAX);", "return (float)((double)a / 480.0);"),
    ("scale: multiply by a rounded reciprocal", "return (float)((double)a / ORA_E4M3_MAX);",
     "return a * (float)(1.0 / ORA_E4M3_MAX);"),
    ("codes: multiply by the rounded reciprocal of the scale",
     "return ora_e4m3_encode((float)((double)x / (double)s));",
     "return ora_e4m3_encode(x * (1.0f / s));"),
    # block quantization
    ("blocks: amax misses the block's last column",
     "for (r = r0; r < r1; r++)\n                for (c = c0; c < c1; c++) {\n                    float a",
     "for (r = r0; r < r1; r++)\n                for (c = c0; c < c1 - 1; c++) {\n                    float a"),
    ("blocks: amax misses the block's last row",
     "for (r = r0; r < r1; r++)\n                for (c = c0; c < c1; c++) {\n                    float a",
     "for (r = r0; r < (r1 - r0 > 1 ? r1 - 1 : r1); r++)\n                for (c = c0; c < c1; c++) {\n"
     "                    float a"),
    ("blocks: amax without fabs", "float a = fabsf(bf16_bits_to_float(x[r * cols + c]));",
     "float a = bf16_bits_to_float(x[r * cols + c]);"),
    ("blocks: scale strides swapped", "s[rb * s_stride_r + cb * s_stride_c] = scale;",
     "s[rb * s_stride_c + cb * s_stride_r] = scale;"),
    ("per tensor: amax misses the last element", "for (i = 0; i < n; i++) {\n        float a",
     "for (i = 0; i + 1 < n; i++) {\n        float a"),
    # GEMM
    ("gemm: first K term dropped", "for (k = 0; k < K; k++) {\n        double a = (double)sa",
     "for (k = 1; k < K; k++) {\n        double a = (double)sa"),
    ("gemm: weight K index reversed", "ora_e4m3_decode(qw[n * K + k]);\n        acc",
     "ora_e4m3_decode(qw[n * K + (K - 1 - k)]);\n        acc"),
    ("gemm: weight scale of the wrong K block", "(double)sw[(n / bn) * kb_count + k / bk]",
     "(double)sw[(n / bn) * kb_count + (kb_count - 1 - k / bk)]"),
    ("gemm: activation scale of the wrong row", "(double)sa[(k / gk) * lda_s + m]",
     "(double)sa[(k / gk) * lda_s + (lda_s - 1 - m)]"),
    ("gemm: weight scale ignored", "double b = (double)sw[(n / bn) * kb_count + k / bk] * ora_e4m3_decode",
     "double b = 1.0 * ora_e4m3_decode"),
    ("gemm: magnitude sum without abs", "mag += fabs(a * b);\n    }\n    *y = acc;", "mag += a * b;\n    }\n    *y = acc;"),
    ("gemm: subtracted product", "acc += a * b;\n        mag += fabs(a * b);\n    }\n    *y",
     "acc -= a * b;\n        mag += fabs(a * b);\n    }\n    *y"),
    ("grouped: expert range closed at the top", "if (ms[i] >= offsets[e] && ms[i] < offsets[e + 1])",
     "if (ms[i] >= offsets[e] && ms[i] <= offsets[e + 1])"),
    ("grouped: first row of an expert given to the previous one",
     "if (ms[i] >= offsets[e] && ms[i] < offsets[e + 1])\n                expert = e;",
     "if (ms[i] >= offsets[e] && ms[i] <= offsets[e + 1] && ms[i] < offsets[num_groups] && expert < 0)\n"
     "                expert = e;"),
    ("grouped: weight scales of expert 0 for every expert", "sw + expert * nb_count * kb_count", "sw"),
    ("per-tensor gemm: activation scale dropped", "double a = (double)sa * ora_e4m3_decode(qa[m * K + k]);",
     "double a = ora_e4m3_decode(qa[m * K + k]);"),
    ("per-tensor gemm: weight scale dropped", "double b = (double)sw * ora_e4m3_decode(qw[n * K + k]);",
     "double b = ora_e4m3_decode(qw[n * K + k]);"),
    ("points: rows paired with another point's column", "qw, sw, K, gk, bn, bk, ms[i], ns[i],",
     "qw, sw, K, gk, bn, bk, ms[i], ns[npts - 1 - i],"),
    ("per-tensor points: weight row of another point", "qa + ms[i] * K, sa, qw + ns[i] * K, sw,",
     "qa + ms[i] * K, sa, qw + ns[npts - 1 - i] * K, sw,"),
    ("grouped: expert 0's weights for every expert", "qw + expert * N * K", "qw"),
    # BF16 rounding and the FP8 KV cache
    ("bf16: ties away from zero", "r = nearbyint(a / quantum) * quantum;", "r = round(a / quantum) * quantum;"),
    ("bf16: seven significant bits", "quantum = ldexp(1.0, exponent - 7);", "quantum = ldexp(1.0, exponent - 6);"),
    ("bf16: subnormal spacing one binade too fine", "if (exponent < -126)\n        exponent = -126;",
     "if (exponent < -127)\n        exponent = -127;"),
    ("kv store: last element of each row skipped",
     "for (e = 0; e < elems; e++)\n            cache[slots[t] * elems + e]",
     "for (e = 0; e + 1 < elems; e++)\n            cache[slots[t] * elems + e]"),
    ("kv store: scale taken as its reciprocal",
     "cache[slots[t] * elems + e] = quant_value(bf16_bits_to_float(x[t * elems + e]), scale);",
     "cache[slots[t] * elems + e] = quant_value(bf16_bits_to_float(x[t * elems + e]), 1.0f / scale);"),
    ("kv load: rows of the mirrored slot", "ora_e4m3_decode(cache[slots[t] * elems + e])",
     "ora_e4m3_decode(cache[(num_slots - 1 - slots[t]) * elems + e])"),
    ("kv load: scale ignored", "(double)scale));", "1.0));"),
    ("static quantization: scale taken as its reciprocal",
     "q[i] = quant_value(bf16_bits_to_float(x[i]), scale);",
     "q[i] = quant_value(bf16_bits_to_float(x[i]), 1.0f / scale);"),
]


def _tree(tmp, name: str, source: str) -> str:
    root = os.path.join(tmp, name)
    os.makedirs(os.path.join(root, "tests"))
    shutil.copytree(os.path.join(ROOT, "synth"), os.path.join(root, "synth"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    os.makedirs(os.path.join(root, "oracle"))
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), os.path.join(root, "oracle"))
    with open(os.path.join(root, "oracle", "fp8_oracle.c"), "w") as f:
        f.write(source)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(root, "tests", "golden"))
    for f in ["conftest.py"] + PIN_FILES:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(root, "tests"))
    return root


def _run_pins(root: str) -> subprocess.CompletedProcess:
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    check = ("import oracle, sys; assert oracle.__file__.startswith(sys.argv[1]), oracle.__file__")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-rf", "-p", "no:cacheprovider", "--rootdir", root,
           *[os.path.join(root, "tests", f) for f in PIN_FILES]]
    # Prove the copy's oracle is the one imported, then run the pins.
    subprocess.run([sys.executable, "-c", check, root], cwd=root, env=env, check=True,
                   capture_output=True, text=True)
    return subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    with open(os.path.join(ROOT, "oracle", "fp8_oracle.c")) as f:
        original = f.read()
    tmp = str(tmp_path_factory.mktemp("mutants"))
    jobs = {"unmutated": _tree(tmp, "m00", original)}
    for i, (name, old, new) in enumerate(MUTANTS, 1):
        assert original.count(old) == 1, f"{name}: snippet must occur exactly once"
        jobs[name] = _tree(tmp, f"m{i:02d}", original.replace(old, new))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as pool:
        results = dict(zip(jobs, pool.map(_run_pins, jobs.values())))
    return results


def test_unmutated_copy_passes_its_pins(outcomes):
    r = outcomes["unmutated"]
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(outcomes, name):
    r = outcomes[name]
    # Exit code 1: a pin failed (2 would be an interruption or a collection error).
    assert r.returncode == 1, f"{name} survived the pins:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
