"""The oracle's pins catch plausible mistakes in it.

Each case plants one mistake -- a dropped term, a wrong sign, index or
operand order, an off-by-one, a wrong formula -- in a scratch copy of
oracle.c, rebuilds that copy, and runs the pin suite (test_oracle_pins.py)
against it: the suite must fail.  A control copy without a mistake must
pass, so a failure means the pins caught the planted mistake and not that
the scratch setup broke.  The repository's own oracle is never modified.
CPU only; the copies run four at a time (well under a minute).
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in oracle.c, replacement); each text occurs exactly once
MUTATIONS = [
    ("conv_output_size", "*Ho = H - 3 + 1;", "*Ho = H - 3;"),
    ("pool_ceil_mode", "return (Ho - k) / k + 1;", "return (Ho + k - 1) / k;"),
    ("conv_taps_swapped", "(i + kh)) * W + (j + kw)", "(i + kw)) * W + (j + kh)"),
    ("conv_bias_dropped", "double acc = (double)b[co];", "double acc = 0.0;"),
    ("filter_taps_transposed", "* 9 + kh * 3 + kw]", "* 9 + kw * 3 + kh]"),
    ("filter_channels_swapped", "w[((int64_t)co * Cin + ci) * 9", "w[((int64_t)ci * Cin + co % Cin) * 9"),
    ("max_instead_of_min", "if (am < 0 || v < m) {", "if (am < 0 || v > m) {"),
    ("ties_keep_last_channel", "if (am < 0 || v < m) {", "if (am < 0 || v <= m) {"),
    ("one_tanh", "if (tanh2) m = tanh(tanh(m));", "if (tanh2) m = tanh(m);"),
    ("min_scalar_dropped", "double v = scalar * ycol[(int64_t)c * cstride];", "double v = ycol[(int64_t)c * cstride];"),
    ("lrelu_slope_on_positives", "v = (v > 0.0 ? v : 0.0) + slope * (v < 0.0 ? v : 0.0);",
     "v = slope * (v > 0.0 ? v : 0.0) + (v < 0.0 ? v : 0.0);"),
    ("gelu_wrong_scale", "erf(v / sqrt(2.0))", "erf(v / 2.0)"),
    ("gelu_tanh_form", "0.5 * v * (1.0 + erf(v / sqrt(2.0)))",
     "0.5 * v * (1.0 + tanh(0.7978845608028654 * (v + 0.044715 * v * v * v)))"),
    ("multiplier_dropped", "double v = y * mult;", "double v = y;"),
    ("gn_unbiased_variance", "double var = ss / (double)cnt;", "double var = ss / (double)(cnt - 1);"),
    ("gn_eps_outside_sqrt", "1.0 / sqrt(var + c->eps)", "1.0 / (sqrt(var) + c->eps)"),
    ("gn_affine_order", "((v - mean) * rstd * (double)c->gamma[ch] + (double)c->beta[ch]) * (double)c->scale[ch]",
     "((v - mean) * rstd + (double)c->beta[ch]) * (double)c->gamma[ch] * (double)c->scale[ch]"),
    ("gn_beta_dropped", "+ (double)c->beta[ch]) * (double)c->scale[ch]", ") * (double)c->scale[ch]"),
    ("gn_stats_miss_last_row", "for (int64_t k = 0; k < cnt; ++k) s += yg[k];",
     "for (int64_t k = 0; k < cnt - Wo; ++k) s += yg[k];"),
    ("pool_window_shifted", "(pw * k + bb)]", "(pw * k + bb + (pw + 1 < Wp))]"),
    ("pool_min_instead_of_max", "if (barg < 0 || v > best) {", "if (barg < 0 || v < best) {"),
    ("clamp_low_to_high", "if (o < c->clamp_lo) o = c->clamp_lo;", "if (o < c->clamp_lo) o = c->clamp_hi;"),
    ("clamp_high_dropped", "if (o > c->clamp_hi) o = c->clamp_hi;", ""),
]


def _scratch_copy(base, name):
    dst = os.path.join(base, name)
    ignore = shutil.ignore_patterns("_build", "__pycache__", "*.so")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"), ignore=ignore)
    shutil.copytree(os.path.join(ROOT, "synth"), os.path.join(dst, "synth"), ignore=ignore)
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    return dst


def _run_pins(base, name, old, new):
    dst = _scratch_copy(base, name)
    src = os.path.join(dst, "oracle", "oracle.c")
    text = open(src).read()
    if old is not None:
        assert text.count(old) == 1, f"{name}: the text to change must occur once"
        with open(src, "w") as f:
            f.write(text.replace(old, new))
    env = dict(os.environ, PYTHONPATH=dst, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q", "-p",
                        "no:cacheprovider"], cwd=dst, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    base = str(tmp_path_factory.mktemp("oracle_mutants"))
    cases = [("control", None, None)] + MUTATIONS
    with ThreadPoolExecutor(max_workers=4) as ex:
        futs = {name: ex.submit(_run_pins, base, name, old, new) for name, old, new in cases}
        return {name: f.result() for name, f in futs.items()}


def test_control_copy_passes(outcomes):
    rc, out = outcomes["control"]
    assert rc == 0, out


@pytest.mark.parametrize("name", [m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(outcomes, name):
    rc, out = outcomes[name]
    assert rc == 1, f"{name}: the pins did not fail (exit {rc})\n{out}"
