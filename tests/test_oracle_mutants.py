"""The oracle's pins have teeth: each plausible mistake below, planted in a private copy of
the oracle's C source and compiled on the CPU, must make at least one pin fail."""
import json
import os
import subprocess
import sys

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_golden as golden
from tests import test_oracle_refine_pins as refine_pins

MUTANTS = {
    "dropped_scale": ("z[j] = dot * scale;", "z[j] = dot;"),
    "transposed_key_index": ("const uint16_t *kr = k + (size_t)r * D;",
                             "const uint16_t *kr = k + (size_t)r;"),
    "normaliser_without_max_shift": ("z[j] = exp(z[j] - zmax);\n            sum += z[j];",
                                     "sum += exp(z[j]);\n            z[j] = exp(z[j] - zmax);"),
    "merge_drops_rescale": ("L += exp(m[c] - M) * l[c];", "L += l[c];"),
    "evidence_not_averaged": ("f[j] = s / (double)G;", "f[j] = s;"),
    "tie_break_to_higher_index": ("return (x->idx > y->idx) - (x->idx < y->idx);",
                                  "return (x->idx < y->idx) - (x->idx > y->idx);"),
    "prior_distance_off_by_one": ("const int d = (L - W) - j;\n        float rt = (float)d * inv_tau;\n        if (rt > 1.0f)\n            rt = 1.0f;\n        const float a",
                                  "const int d = (L - W) - j - 1;\n        float rt = (float)d * inv_tau;\n        if (rt > 1.0f)\n            rt = 1.0f;\n        const float a"),
    "prior_wrong_sign": ("const float b = c2 * rt;\n        s[i] = a + b;", "const float b = -c2 * rt;\n        s[i] = a + b;"),
    "window_off_by_one": ("int w0 = L_now - W;", "int w0 = L_now - W + 1;"),
    "candidates_include_window": ("const int n = L - W - S;", "const int n = L - S;"),
    "tmax_strict": ("mask[t - 1] || (t_max > 0 && t - last >= t_max)",
                    "mask[t - 1] || (t_max > 0 && t - last > t_max)"),
    "first_step_not_slow": ("int s = (t == 0) || mask[t - 1]", "int s = (t < 0) || mask[t - 1]"),
    "token_trigger_off_by_one": ("if (tokens[t - 1] == trigger_ids[i])",
                                 "if (tokens[t] == trigger_ids[i])"),
    "nms_non_strict": ("if (!(w > v))", "if (!(w >= v))"),
    "nms_similarity_ignored": ("return delta <= 0.0f || w - v <= delta;", "return 1;"),
    "nms_similarity_reversed": ("return delta <= 0.0f || w - v <= delta;",
                                "return delta <= 0.0f || w - v >= delta;"),
    "exclusivity_wrong_sign": ("s[(size_t)h * n + i] = v - pen;", "s[(size_t)h * n + i] = v + pen;"),
    "geometric_weights_swapped": ("const float a = c1 * sfi_oracle_log2f(fj);",
                                  "const float a = lam_f * sfi_oracle_log2f(fj);"),
    "key_norm_term_inverted": ("float g = nu / knorm[(size_t)h * L + j];",
                               "float g = knorm[(size_t)h * L + j] / nu;"),
    "log2_series_term_dropped": ("s = s * t2 + 0x1.99999ap-3f;", "s = s * t2;"),
}

PIN_TESTS = [(pins, name) for name in dir(pins) if name.startswith("test_")] + \
    [(refine_pins, name) for name in dir(refine_pins) if name.startswith("test_")] + \
    [(golden, name) for name in dir(golden) if name.startswith("test_")]


def run_pins():
    """Run every pin (with its parametrisations); return the names that failed."""
    import inspect
    failed = []
    for mod, name in PIN_TESTS:
        fn = getattr(mod, name)
        marks = getattr(fn, "pytestmark", [])
        cases = [{}]
        for m in marks:
            if m.name == "parametrize":
                argnames, values = m.args[0], m.args[1]
                argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else argnames
                cases = [dict(c, **dict(zip(argnames, v if isinstance(v, (tuple, list)) else (v,))))
                         for c in cases for v in values]
        for kw in cases:
            try:
                fn(**kw)
            except Exception:
                failed.append(name)
                break
    return failed


@pytest.fixture(scope="module")
def src():
    with open(os.path.join(os.path.dirname(oracle.__file__), "sfi_oracle.c")) as f:
        return f.read()


def test_unmutated_oracle_passes_all_pins():
    assert run_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, src, tmp_path):
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", so, str(path), "-lm"])
    # A mutant may also corrupt memory; run its pins in a child process so a crash counts
    # as caught without taking the test session down.
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import json, oracle; from tests import test_oracle_mutants as m; "
            f"oracle._lib = oracle.load({so!r}); print(json.dumps(m.run_pins()))")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=600)
    if r.returncode == 0:
        failed = json.loads(r.stdout.strip().splitlines()[-1])
        assert failed, f"no pin caught the planted mistake '{name}'"
