"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (in a
temporary directory, on the CPU), then runs the pin suites against that copy
and expects them to fail.  The mistakes are the kind a restatement of the
pages could make: an off-by-one window, a non-strict gate, the wrong GQA
grouping, a missing square, a dropped softmax term in the gradient, the wrong
sigmoid derivative in the straight-through gate, an inverted decode gate, an
averaged instead of summed divergence, unscaled scores, a subtracted router
bias.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_SUITES = ("test_oracle_pins.py", "test_oracle_backward_pins.py", "test_oracle_anchor_pins.py")

# (name, original text, planted text); the original must occur in the source.
MUTATIONS = [
    ("window_off_by_one", "int64_t a = i - W + 1;", "int64_t a = i - W;"),
    ("gate_not_strict", "gate[t] = acc > 0.0 ? 1 : 0;", "gate[t] = acc >= 0.0 ? 1 : 0;"),
    ("gqa_interleaved", "int64_t kvh = h / (Hq / Hkv);\n    int64_t lo, hi;",
     "int64_t kvh = h % Hkv;\n    int64_t lo, hi;"),
    ("lse_without_max", "if (lse) *lse = mx + log(den);\n}\n\nstatic int shapes_ok",
     "if (lse) *lse = log(den);\n}\n\nstatic int shapes_ok"),
    ("anchored_lse_without_max",
     "if (lse) *lse = mx + log(den);\n}\n\n/* Routed prefill with S global anchors",
     "if (lse) *lse = log(den);\n}\n\n/* Routed prefill with S global anchors"),
    ("mse_not_squared", "acc += e * e;", "acc += fabs(e);"),
    ("softplus_unstable_branch", "log1p(exp(-fabs(x)))", "log1p(exp(-x))"),
    ("gamma_without_alpha", "eps + nll[t] + alpha * mse[t]", "eps + nll[t] + mse[t]"),
    ("grad_drops_row_term", "double ds = p * (dp - D);", "double ds = p * dp;"),
    ("grad_dq_unscaled", "dq[c] += scale * ds * kj[c];", "dq[c] += ds * kj[c];"),
    ("grad_dv_unweighted", "dv[j * kstride + c] += p * dout[c];",
     "dv[j * kstride + c] += dout[c];"),
    ("grad_dk_sign", "dk[j * kstride + c] += scale * ds * q[c];",
     "dk[j * kstride + c] -= scale * ds * q[c];"),
    ("grad_gqa_interleaved", "for (int64_t h = kvh * G; h < (kvh + 1) * G; ++h)",
     "for (int64_t h = kvh; h < Hq; h += Hkv)"),
    ("ste_missing_derivative", "double g = sg * (1.0 - sg) * acc;", "double g = sg * acc;"),
    ("regulariser_wrong_derivative", "g += d_reg[t] * gamma[t] * sg;",
     "g += d_reg[t] * gamma[t] * (1.0 - sg);"),
    ("router_dh_from_logit", "dh[t * D + j] = d_logits[t] * w[j];",
     "dh[t * D + j] = logits[t] * w[j];"),
    ("anchor_off_by_one", "for (int64_t j = 0; j < lo && j < S; ++j) idx[n++] = j;",
     "for (int64_t j = 0; j < lo && j <= S; ++j) idx[n++] = j;"),
    ("anchor_not_causal", "for (int64_t j = 0; j < lo && j < S; ++j) idx[n++] = j;",
     "for (int64_t j = 0; j < S && j < lo + W; ++j) if (j < lo || j > i) idx[n++] = j;"),
    ("decode_gate_inverted", "key_range(gate[b] != 0, (int64_t)seq_lens[b] - 1, W, &lo, &hi);",
     "key_range(gate[b] == 0, (int64_t)seq_lens[b] - 1, W, &lo, &hi);"),
    ("decode_gqa_interleaved", "kvh = h / (Hq / Hkv);\n            int64_t lo, hi;",
     "kvh = h % Hkv;\n            int64_t lo, hi;"),
    ("decode_anchored_gqa_interleaved",
     "kvh = h / (Hq / Hkv);\n            int64_t n = anchored_keys(gate[b] != 0,",
     "kvh = h % Hkv;\n            int64_t n = anchored_keys(gate[b] != 0,"),
    ("prefill_anchored_gqa_interleaved",
     "kvh = h / (Hq / Hkv);\n            int64_t n = anchored_keys(gate[b * N + i] != 0,",
     "kvh = h % Hkv;\n            int64_t n = anchored_keys(gate[b * N + i] != 0,"),
    ("mse_averaged", "*mse = acc;", "*mse = acc / (double)(Hq * d);"),
    ("softplus_missing_max", "return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));",
     "return x + log1p(exp(-fabs(x)));"),
    ("scores_unscaled", "kj = k + (lo + t) * kstride;\n        double dot = 0.0;\n"
     "        for (int64_t c = 0; c < d; ++c) dot += q[c] * kj[c];\n        s[t] = scale * dot;",
     "kj = k + (lo + t) * kstride;\n        double dot = 0.0;\n"
     "        for (int64_t c = 0; c < d; ++c) dot += q[c] * kj[c];\n        s[t] = dot;"),
    ("anchored_scores_unscaled", "kj = k + idx[t] * stride;\n        double dot = 0.0;\n"
     "        for (int64_t c = 0; c < d; ++c) dot += q[c] * kj[c];\n        s[t] = scale * dot;",
     "kj = k + idx[t] * stride;\n        double dot = 0.0;\n"
     "        for (int64_t c = 0; c < d; ++c) dot += q[c] * kj[c];\n        s[t] = dot;"),
    ("router_bias_subtracted", "acc += bias;", "acc -= bias;"),
    ("gamma_without_eps", "eps + nll[t] + alpha * mse[t]", "nll[t] + alpha * mse[t]"),
]


def _plant(tmp_path, original, planted):
    for sub in ("oracle", "tests"):
        os.makedirs(tmp_path / sub, exist_ok=True)
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), tmp_path / "oracle")
    src = open(os.path.join(ROOT, "oracle", "swiattn_oracle.c")).read()
    assert src.count(original) == 1, original
    (tmp_path / "oracle" / "swiattn_oracle.c").write_text(src.replace(original, planted))
    for name in PIN_SUITES + ("conftest.py",):
        shutil.copy(os.path.join(ROOT, "tests", name), tmp_path / "tests")
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")


def _run_pins(where):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1", OMP_NUM_THREADS="2")
    return subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"]
        + [os.path.join("tests", s) for s in PIN_SUITES],
        cwd=where, env=env, capture_output=True, text=True, timeout=600)


def test_unmodified_copy_passes(tmp_path):
    _plant(tmp_path, "int64_t a = i - W + 1;", "int64_t a = i - W + 1;")
    r = _run_pins(tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,original,planted", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, original, planted):
    _plant(tmp_path, original, planted)
    r = _run_pins(tmp_path)
    assert r.returncode == 1, f"{name} survived the pins:\n{r.stdout[-2000:]}"
