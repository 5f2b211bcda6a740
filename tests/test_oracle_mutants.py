"""The oracle's pins must be discriminating: each plausible mistake planted in a copy of
the oracle (a dropped term, a wrong sign, index or operand, a wrong tie rule or constant)
has to make the pin suite fail.  Mutants are built from a temporary copy of the source
and run in a child pytest process, so a crashing mutant cannot take this process down.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ar_oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_oracle_formats.py"),
        os.path.join(ROOT, "tests", "test_oracle_method.py")]

# (name, original text, planted mistake)
MUTANTS = [
    ("rank_order_reversed",
     "float acc = load_elem(partials[0], i, dtype);\n    for (int r = 1; r < n; ++r) acc = acc + load_elem(partials[r], i, dtype);",
     "float acc = load_elem(partials[n - 1], i, dtype);\n    for (int r = n - 2; r >= 0; --r) acc = acc + load_elem(partials[r], i, dtype);"),
    ("binary64_accumulator", "float acc = load_elem(partials[0], i, dtype);",
     "double acc = load_elem(partials[0], i, dtype);"),
    ("residual_dropped", "float zv = sv + load_elem(res_in, base + j, dtype);", "float zv = sv;"),
    ("residual_sign", "float zv = sv + load_elem(res_in, base + j, dtype);",
     "float zv = sv - load_elem(res_in, base + j, dtype);"),
    ("eps_outside_sqrt", "1.0 / sqrt(mean_sq + (double)eps)", "1.0 / (sqrt(mean_sq) + (double)eps)"),
    ("mean_over_h_minus_1", "sumsq / (double)h", "sumsq / (double)(h > 1 ? h - 1 : 1)"),
    ("abs_instead_of_square", "sumsq += zv * zv;", "sumsq += fabs(zv);"),
    ("gemma_ignored", "gemma ? 1.0 + wv : wv", "wv"),
    ("gemma_sign", "gemma ? 1.0 + wv : wv", "gemma ? 1.0 - wv : wv"),
    ("norm_reads_sum_not_residual_sum",
     "double zv = (double)load_elem(z_row, j, dtype);\n    double wv",
     "double zv = (double)load_elem(s, base + j, dtype);\n    double wv"),
    ("fp8_max_240", "  float sc = amax / 448.0f;\n  scale[row] = sc;", "  float sc = amax / 240.0f;\n  scale[row] = sc;"),
    ("scale_row_index", "scale[row] = sc;", "scale[0] = sc;"),
    ("quant_of_unrounded_z", "if (quant) quant_row(q + base, scale + r, y_row, 0, h, dtype);",
     "if (quant) quant_row(q + base, scale + r, z_row, 0, h, dtype);"),
    ("ties_away_from_zero", "return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    ("no_gradual_underflow", "  if (e < emin) e = emin;\n", "\n"),
    ("e4m3_overflow_to_nan", "if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);",
     "if (a >= 464.0) return (uint8_t)(sign | 0x7Fu);"),
    ("bf16_bias", "encode_fields(r, 8, -126, 127)", "encode_fields(r, 8, -126, 126)"),
    ("f16_max_finite_overflows", "if (r >= 65536.0)", "if (r >= 65504.0)"),
    ("row_stride", "int gemma, int skip_norm, int dtype) {\n  int64_t base = row * h;",
     "int gemma, int skip_norm, int dtype) {\n  int64_t base = row * (h > 1 ? h - 1 : 1);"),
    ("fp32_output_drops_weight", "if (y32) y32[base + j] = (float)yv;",
     "if (y32) y32[base + j] = (float)(zv * inv_rms);"),
    ("fp32_output_via_16bit", "if (y32) y32[base + j] = (float)yv;",
     "if (y32) y32[base + j] = (float)zv * (float)inv_rms * (float)factor;"),
    ("skip_norm_outputs_the_sum", "if (y32) y32[base + j] = load_elem(z_row, j, dtype);",
     "if (y32) y32[base + j] = load_elem(s, base + j, dtype);"),
    ("skip_norm_still_normalises", "  if (skip_norm) {\n", "  if (0) {\n"),
    ("group_bounds_off_by_one", "const int64_t j0 = k * g, j1 = j0 + g;", "const int64_t j0 = k * g, j1 = j0 + g - 1;"),
    ("group_scale_index", "scale + r * (h / group), (const uint16_t*)y + r * h", "scale + r, (const uint16_t*)y + r * h"),
    ("group_max_448_240", "    float sc = amax / 448.0f;\n    scale[k] = sc;", "    float sc = amax / 240.0f;\n    scale[k] = sc;"),
    ("fp8_quotient_by_reciprocal", "float v = load_elem(y, base + j, dtype) / sc;",
     "float v = load_elem(y, base + j, dtype) * (1.0f / sc);"),
    ("fp8_scale_flushes_subnormals", "  float sc = amax / 448.0f;\n  scale[row] = sc;",
     "  float sc = amax / 448.0f;\n  if (sc < 1.17549435e-38f) sc = 0.0f;\n  scale[row] = sc;"),
]


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


def _run_pins(lib):
    env = dict(os.environ, ORACLE_LIB=lib)
    env.pop("PYTEST_ADDOPTS", None)
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def _build(tmp_path, text, name):
    import oracle
    d = tmp_path / name
    d.mkdir()
    shutil.copy(os.path.join(ROOT, "oracle", "ar_oracle.h"), d / "ar_oracle.h")
    (d / "ar_oracle.c").write_text(text)
    return oracle.build(str(d / "ar_oracle.c"), str(d / "liboracle.so"))


def test_unmutated_copy_passes(tmp_path, src_text):
    lib = _build(tmp_path, src_text, "control")
    r = _run_pins(lib)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, src_text, name, old, new):
    assert src_text.count(old) == 1, f"mutation site for {name} not found exactly once"
    lib = _build(tmp_path, src_text.replace(old, new), name)
    r = _run_pins(lib)
    assert r.returncode != 0, f"planted mistake {name} passed every pin"
