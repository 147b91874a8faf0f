"""The oracle's pins catch plausible mistakes: each case plants one mistake in a
temporary copy of the oracle (the C recurrence or the Python input steps), runs the
pin suites against that copy in a subprocess, and requires at least one pin to fail.
The unchanged copy must pass, so a failure is the planted mistake's doing.

The mistakes follow the steps of the recurrence of "Kimi Delta Attention (KDA)"
(brain.bigb.es, the five-line reference recurrence: forget, predict, correct,
rank-one write, read after the write, with the d_k^-1/2 output scale) and of the
input steps of the DeltaNet forward of "22580: от GPT-2 до Kimi K3" (section
"DeltaNet, или Fast Weight Programmers": silu, L2 norm, sigmoid write strength):
a wrong sign, a dropped factor, a wrong operand, a wrong head or token index, or
two steps in the wrong order.  CPU only; nothing here touches the CUDA library."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C_SRC = "oracle/kda_oracle.c"
PY_SRC = "oracle/__init__.py"
PIN_FILES = ["tests/test_oracle_pins.py", "tests/test_oracle_prep_pins.py"]

# (name, file, text in the oracle, replacement); each text occurs exactly once
REPLACEMENTS = [
    ("forget_sign", C_SRC, "const double a = exp(gt[i]);", "const double a = exp(-gt[i]);"),
    ("forget_dropped", C_SRC, "const double a = exp(gt[i]);", "const double a = 1.0 + 0.0 * gt[i];"),
    ("predict_with_query", C_SRC, "pred += S[(size_t)i * dv + j] * kt[i];",
     "pred += S[(size_t)i * dv + j] * qt[i];"),
    ("correction_sign", C_SRC, "e[j] = bt * (vt[j] - pred);", "e[j] = bt * (vt[j] + pred);"),
    ("write_strength_dropped", C_SRC, "e[j] = bt * (vt[j] - pred);", "e[j] = (vt[j] - pred);"),
    ("write_halved", C_SRC, "S[(size_t)i * dv + j] += kt[i] * e[j];",
     "S[(size_t)i * dv + j] += 0.5 * kt[i] * e[j];"),
    ("write_along_query", C_SRC, "S[(size_t)i * dv + j] += kt[i] * e[j];",
     "S[(size_t)i * dv + j] += qt[i] * e[j];"),
    ("read_with_key", C_SRC, "acc += S[(size_t)i * dv + j] * qt[i];",
     "acc += S[(size_t)i * dv + j] * kt[i];"),
    ("output_scale_dropped", C_SRC, "ot[j] = J->scale * acc;", "ot[j] = acc;"),
    ("last_token_dropped", C_SRC, "for (int64_t t = bos; t < eos; ++t) {",
     "for (int64_t t = bos; t < eos - 1; ++t) {"),
    ("initial_state_ignored", C_SRC, "if (J->init_state)\n", "if (0 && J->init_state)\n"),
    ("gate_of_head_zero", C_SRC, "const double *gt = J->g + ((size_t)t * H + h) * dk;",
     "const double *gt = J->g + ((size_t)t * H) * dk;"),
    ("write_strength_of_head_zero", C_SRC, "const double bt = J->beta[(size_t)t * H + h];",
     "const double bt = J->beta[(size_t)t * H];"),
    ("silu_sign", PY_SRC, "k = k / (1.0 + np.exp(-k))", "k = k / (1.0 + np.exp(k))"),
    ("sigmoid_sign", PY_SRC, "beta = 1.0 / (1.0 + np.exp(-beta))",
     "beta = 1.0 / (1.0 + np.exp(beta))"),
    ("norm_without_root", PY_SRC,
     "q = q / np.maximum(np.sqrt(np.sum(q * q, axis=-1, keepdims=True)), 1e-12)",
     "q = q / np.maximum(np.sum(q * q, axis=-1, keepdims=True), 1e-12)"),
    ("norm_over_tokens", PY_SRC,
     "k = k / np.maximum(np.sqrt(np.sum(k * k, axis=-1, keepdims=True)), 1e-12)",
     "k = k / np.maximum(np.sqrt(np.sum(k * k, axis=0, keepdims=True)), 1e-12)"),
]

# the loop body's steps, each starting at its comment; the last ends the loop
STEP_MARKS = ["    /* forget", "    /* predict + correct", "    /* write:", "    /* read after write",
              "  }\n  if (J->final_state)"]
SWAPS = [("predict_before_forget", 0), ("read_before_write", 2)]


def _swap_steps(text, first):
    """Exchange step `first` and step `first + 1` of the per-token loop."""
    cuts = [text.index(m) for m in STEP_MARKS]
    a, b, c = cuts[first], cuts[first + 1], cuts[first + 2]
    return text[:a] + text[b:c] + text[a:b] + text[c:]


def _copy_tree(dst):
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    for name in ["conftest.py"] + [os.path.basename(f) for f in PIN_FILES]:
        shutil.copy(os.path.join(ROOT, "tests", name), os.path.join(dst, "tests", name))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), os.path.join(dst, "pytest.ini"))


def _run_pins(dst):
    env = dict(os.environ)
    env.pop("PYTHONPATH", None)  # the copy's oracle, not the repository's
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          *PIN_FILES], cwd=dst, env=env, capture_output=True, text=True,
                         timeout=600)
    return res.returncode, res.stdout[-2000:] + res.stderr[-2000:]


def _mutate(dst, name):
    for n, rel, old, new in REPLACEMENTS:
        if n == name:
            path = os.path.join(dst, rel)
            text = open(path, encoding="utf-8").read()
            assert text.count(old) == 1, f"{name}: the oracle text to change is not unique"
            open(path, "w", encoding="utf-8").write(text.replace(old, new))
            return
    first = dict(SWAPS)[name]
    path = os.path.join(dst, C_SRC)
    text = open(path, encoding="utf-8").read()
    open(path, "w", encoding="utf-8").write(_swap_steps(text, first))


def _case(tmp, name):
    dst = os.path.join(tmp, name)
    _copy_tree(dst)
    if name != "unchanged":
        _mutate(dst, name)
    return name, _run_pins(dst)


NAMES = [r[0] for r in REPLACEMENTS] + [s[0] for s in SWAPS]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        return dict(ex.map(lambda n: _case(tmp, n), ["unchanged"] + NAMES))


def test_unchanged_copy_passes_its_pins(outcomes):
    rc, log = outcomes["unchanged"]
    assert rc == 0, log


@pytest.mark.parametrize("name", NAMES)
def test_planted_mistake_fails_a_pin(outcomes, name):
    rc, log = outcomes[name]
    assert rc == 1 and "failed" in log, f"{name} was not caught:\n{log}"
