"""Plants one mistake at a time in a copy of the oracle (on the CPU) and checks that the
pins reject every such copy: test_oracle_pins.py for the forward, test_oracle_backward_pins.py
for the backward, and the full-attention, masked-variant and block-front-end pins for theirs."""
import inspect

import pytest

import oracle
import tests.test_oracle_backward_pins as bpins
import tests.test_oracle_block_pins as blpins
import tests.test_oracle_causal_pins as cpins
import tests.test_oracle_full_attention_pins as fpins
import tests.test_oracle_pins as pins

# (name, text in anchor_oracle.c, replacement): each a plausible slip.
MUTANTS = [
    ("scale dropped", "a[j] = scale * s;", "a[j] = s;"),
    ("scale applied twice", "a[j] = scale * s;", "a[j] = scale * scale * s;"),
    ("max subtracted with wrong sign", "a[j] = exp(a[j] - mx);", "a[j] = exp(mx - a[j]);"),
    ("row not normalised", "for (long j = 0; j < m; ++j) a[j] /= z;", ";"),
    ("Delta^-1 dropped", "Wp[j * d + k] = delta[j] != 0.0 ? s / delta[j] : 0.0;", "Wp[j * d + k] = s;"),
    ("Delta from the first token only", "for (long i = 0; i < n; ++i) s += A[i * m + j];", "s = A[j];"),
    ("value column reversed", "s += A[i * m + j] * V[i * d + k];", "s += A[i * m + j] * V[i * d + (d - 1 - k)];"),
    ("first anchor dropped in the apply", "for (long j = 0; j < m; ++j) s += a[j] * Wp[j * d + k];",
     "for (long j = 1; j < m; ++j) s += a[j] * Wp[j * d + k];"),
    ("anchors indexed by batch", "U + (size_t)h * (size_t)m * (size_t)d", "U + (size_t)((b + h) % heads) * (size_t)m * (size_t)d"),
    ("query/anchor dims crossed", "s += Q[i * d + k] * U[j * d + k];", "s += Q[i * d + k] * U[k % m * d + j % d];"),
]


# slips in the backward
BACKWARD_MUTANTS = [
    ("dDelta term dropped", "double g = ddelta[j];", "double g = 0.0;"),
    ("softmax Jacobian with the wrong sign", "G[j] = a[j] * (G[j] - ag);", "G[j] = a[j] * (G[j] + ag);"),
    ("softmax Jacobian without the row term", "G[j] = a[j] * (G[j] - ag);", "G[j] = a[j] * G[j];"),
    ("scale dropped from dQ", "dQ[i * d + k] = scale * s;", "dQ[i * d + k] = s;"),
    ("dU from V instead of Q", "dU[j * d + k] += scale * G[j] * Q[i * d + k];", "dU[j * d + k] += scale * G[j] * V[i * d + k];"),
    ("Delta^-1 dropped from dW", "dW[j * d + k] = delta[j] != 0.0 ? dWp[j * d + k] / delta[j] : 0.0;",
     "dW[j * d + k] = dWp[j * d + k];"),
    ("dDelta with the wrong sign", "ddelta[j] = delta[j] != 0.0 ? -s / (delta[j] * delta[j]) : 0.0;",
     "ddelta[j] = delta[j] != 0.0 ? s / (delta[j] * delta[j]) : 0.0;"),
    ("path through W dropped", "g += dH[i * d + k] * Wp[j * d + k] + V[i * d + k] * dW[j * d + k];",
     "g += dH[i * d + k] * Wp[j * d + k];"),
    ("dV from dW' instead of dW", "for (long j = 0; j < m; ++j) s += a[j] * dW[j * d + k];",
     "for (long j = 0; j < m; ++j) s += a[j] * dWp[j * d + k];"),
    ("dU not summed over the batch", "for (long i = 0; i < heads * m * d; ++i) dU[i] = 0.0;\n    for (long b = 0; b < B; ++b) {",
     "for (long b = 0; b < B; ++b) {\n        for (long i = 0; i < heads * m * d; ++i) dU[i] = 0.0;"),
]


# slips in the full attention of the approximation-error diagnostic
FULL_MUTANTS = [
    ("full: max subtracted with the wrong sign", "p[j] = exp(p[j] - mx);", "p[j] = exp(mx - p[j]);"),
    ("full: not normalised", "H[i * d + k] = s / z;", "H[i * d + k] = s;"),
    ("full: scale dropped", "p[j] = scale * s;\n            if (p[j] > mx) mx = p[j];\n        }\n        double z = 0.0;\n        for (long j = 0; j < nk; ++j) {",
     "p[j] = s;\n            if (p[j] > mx) mx = p[j];\n        }\n        double z = 0.0;\n        for (long j = 0; j < nk; ++j) {"),
    ("full: keys indexed per batch entry", "K + (size_t)h * (size_t)n * (size_t)d", "K + (size_t)((b + h) % heads) * (size_t)n * (size_t)d"),
]


# slips in the masked (causal) variant
CAUSAL_MUTANTS = [
    ("causal: anchor degree counted twice", "delta[l] += a[l];", "delta[l] += 2.0 * a[l];"),
    ("causal: summaries from the first token's value", "W[l * d + k] += a[l] * V[i * d + k];",
     "W[l * d + k] += a[l] * V[k];"),
    ("causal: row weights of the previous token", "if (delta[l] != 0.0) s += a[l] * W[l * d + k] / delta[l];",
     "if (delta[l] != 0.0) s += A[(i > 0 ? i - 1 : 0) * m + l] * W[l * d + k] / delta[l];"),
]


# slips in the block front end (the Q and V projections)
BLOCK_MUTANTS = [
    ("block: Q projected with the value weights", "sq += X[i * dm + c] * Wq[k * dm + c];",
     "sq += X[i * dm + c] * Wv[k * dm + c];"),
    ("block: query weights read transposed", "sq += X[i * dm + c] * Wq[k * dm + c];",
     "sq += X[i * dm + c] * Wq[(c % d) * dm + (k * dm + c) / d % dm];"),
    ("block: head offset of the weights dropped", "const size_t woff = (size_t)h * (size_t)d * (size_t)dm;",
     "const size_t woff = 0;"),
    ("block: batch offset of the tokens dropped", "const size_t xoff = (size_t)b * (size_t)n * (size_t)dm;",
     "const size_t xoff = 0;"),
    ("block: last embedding column skipped", "for (long c = 0; c < dm; ++c) {", "for (long c = 0; c + 1 < dm; ++c) {"),
]


def _run_module_pins(module, mut) -> list:
    import inspect as _inspect
    failed = []
    for name, fn in _inspect.getmembers(module, _inspect.isfunction):
        if name.startswith("test_"):
            try:
                fn(mut)
            except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
                failed.append(name)
    return failed


def _run_bpins(mut) -> list:
    failed = []
    for name, fn in inspect.getmembers(bpins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        cases = [{}]
        if "shape" in params:  # the finite-difference pin on its smallest shape keeps this quick
            cases = [{"shape": (1, 1, 5, 3, 4), "scale": 0.5, "qscale": 1.0}]
        for kw in cases:
            try:
                fn(mut, **kw)
            except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
                failed.append(name)
    return failed


def _run_pins(mut) -> list:
    failed = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or name == "test_bad_arguments_raise":
            continue
        params = inspect.signature(fn).parameters
        cases = [{}]
        if "case" in params:
            cases = [{"case": c} for c in ("m1", "identical_anchors", "zero_queries")]
        for kw in cases:
            try:
                fn(mut, **kw)
            except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
                failed.append(name)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(tmp_path, name, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    mut = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    assert _run_pins(mut), f"no pin rejects the planted mistake '{name}'"


@pytest.mark.parametrize("name,old,new", BACKWARD_MUTANTS, ids=[m[0] for m in BACKWARD_MUTANTS])
def test_backward_pins_reject_planted_mistake(tmp_path, name, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    mut = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    failed = _run_bpins(mut)
    assert failed, f"no backward pin rejects the planted mistake '{name}'"


@pytest.mark.parametrize("name,old,new", FULL_MUTANTS, ids=[m[0] for m in FULL_MUTANTS])
def test_full_attention_pins_reject_planted_mistake(tmp_path, name, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    mut = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    assert _run_module_pins(fpins, mut), f"no full-attention pin rejects the planted mistake '{name}'"


@pytest.mark.parametrize("name,old,new", CAUSAL_MUTANTS, ids=[m[0] for m in CAUSAL_MUTANTS])
def test_causal_pins_reject_planted_mistake(tmp_path, name, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    mut = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    assert _run_module_pins(cpins, mut), f"no causal pin rejects the planted mistake '{name}'"


@pytest.mark.parametrize("name,old,new", BLOCK_MUTANTS, ids=[m[0] for m in BLOCK_MUTANTS])
def test_block_pins_reject_planted_mistake(tmp_path, name, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    mut = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    assert _run_module_pins(blpins, mut), f"no block pin rejects the planted mistake '{name}'"
