"""Mutation check of the oracle's pins (CPU only).

Each case copies ``oracle/ss_oracle.c``, plants ONE plausible mistake (a
dropped term, a wrong sign, an off-by-one index, a swapped operand), compiles
the copy into a temporary library and runs every pin from ``oracle_pins``
against it.  The test passes only if at least one pin fails on the mutant --
i.e. the pins would have caught that mistake in the real oracle.
"""

import os

import numpy as np
import pytest

import oracle
import oracle_pins as P

# (label, text in ss_oracle.c, replacement, which occurrence [0-based])
MUTANTS = [
    ("fwd: D term dropped", "if (p->D) acc += p->D[d] * ut;", "", 0),
    ("fwd: exponent sign", "double a = exp(dt * p->A[at_dn(p, d, n)]);", "double a = exp(-dt * p->A[at_dn(p, d, n)]);", 0),
    ("fwd: decay dropped", "h[n] = a * h[n] + dt", "h[n] = h[n] + dt", 0),
    ("fwd: B read as C", "h[n] = a * h[n] + dt * p->B[at_bln(p, b, t, n)] * ut;",
     "h[n] = a * h[n] + dt * p->C[at_bln(p, b, t, n)] * ut;", 0),
    ("fwd: C read at t-1", "acc += h[n] * p->C[at_bln(p, b, t, n)];",
     "acc += h[n] * p->C[at_bln(p, b, t > 0 ? t - 1 : 0, n)];", 0),
    ("fwd: Delta_t missing from input term", "h[n] = a * h[n] + dt * p->B", "h[n] = a * h[n] + p->B", 0),
    ("bias ignored", "if (p->bias) x += p->bias[d];", "", 0),
    ("softplus: x term dropped", "return x > 0.0 ? x + log1p(exp(-x))", "return x > 0.0 ? log1p(exp(-x))", 0),
    ("softplus: exp instead", ": log1p(exp(x)); }", ": exp(x); }", 0),
    ("silu: sigmoid only", "static double silu_f64(double z) { return z * sigmoid_f64(z); }",
     "static double silu_f64(double z) { return sigmoid_f64(z); }", 0),
    ("last_state from h_{L-2}", "for (int64_t n = 0; n < p->N; n++) last[n] = h[n];",
     "for (int64_t n = 0; n < p->N; n++) last[n] = h[n] - p->B[at_bln(p, b, p->L - 1, n)] * 0.5;", 0),
    ("bwd: recompute uses C as input", "s->h[t * N + n] = a * hprev + dt * p->B[at_bln(p, b, t, n)] * ut;",
     "s->h[t * N + n] = a * hprev + dt * p->C[at_bln(p, b, t, n)] * ut;", 0),
    ("bwd: adjoint uses a_t not a_{t+1}", "double a_next = t + 1 < L ? s->a[(t + 1) * N + n] : 1.0;",
     "double a_next = t + 1 < L ? s->a[t * N + n] : 1.0;", 0),
    ("bwd: adjoint injects B", "double lam = g * Cn + a_next * s->lam[n];", "double lam = g * Bn + a_next * s->lam[n];", 0),
    ("bwd: h_{t-1} read as h_t", "double hprev = t > 0 ? s->h[(t - 1) * N + n] : h_init(p, b, d, n);\n            double a = s->a",
     "double hprev = s->h[t * N + n];\n            double a = s->a", 0),
    ("bwd: du missing Delta", "du_t += lam * dt * Bn;", "du_t += lam * Bn;", 0),
    ("bwd: du missing D*g", "double du_t = p->D ? g * p->D[d] : 0.0;", "double du_t = 0.0;", 0),
    ("bwd: dDelta A-term sign", "dDelta += lam * (p->A[at_dn(p, d, n)] * a * hprev + Bn * ut);",
     "dDelta += lam * (-p->A[at_dn(p, d, n)] * a * hprev + Bn * ut);", 0),
    ("bwd: dDelta missing B*u", "dDelta += lam * (p->A[at_dn(p, d, n)] * a * hprev + Bn * ut);",
     "dDelta += lam * (p->A[at_dn(p, d, n)] * a * hprev);", 0),
    ("bwd: dA missing Delta", "dA[n] += lam * dt * a * hprev;", "dA[n] += lam * a * hprev;", 0),
    ("bwd: dB missing Delta", "dB_acc[at_bln(p, b, t, n)] += lam * dt * ut;", "dB_acc[at_bln(p, b, t, n)] += lam * ut;", 0),
    ("bwd: dC ungated", "dC_acc[at_bln(p, b, t, n)] += g * s->h[t * N + n];",
     "dC_acc[at_bln(p, b, t, n)] += dyt * s->h[t * N + n];", 0),
    ("bwd: dz sign", "(1.0 + zt * (1.0 - sg))", "(1.0 - zt * (1.0 - sg))", 0),
    ("bwd: dz pre-gate misses D", "if (p->D) y0 += p->D[d] * ut;", "", 0),
    ("bwd: softplus grad at Delta", "dDelta * sigmoid_f64(x)", "dDelta * sigmoid_f64(dt)", 0),
    ("bwd: dD ungated", "dD_sum += g * ut;", "dD_sum += dyt * ut;", 0),
    ("bwd: dbias before softplus grad", "dbias_sum += dx;", "dbias_sum += dDelta;", 0),
    ("fwd: h0 ignored", "h[n] = h_init(p, b, d, n);", "h[n] = 0.0;", 0),
    ("bwd: recompute starts from zero", "double hprev = t > 0 ? s->h[(t - 1) * N + n] : h_init(p, b, d, n);\n            double a = exp",
     "double hprev = t > 0 ? s->h[(t - 1) * N + n] : 0.0;\n            double a = exp", 0),
    ("bwd: dA / dDelta at t = 0 without h0", "double hprev = t > 0 ? s->h[(t - 1) * N + n] : h_init(p, b, d, n);\n            double a = s->a",
     "double hprev = t > 0 ? s->h[(t - 1) * N + n] : 0.0;\n            double a = s->a", 0),
    ("bwd: dlast ignored", "s->lam[n] = p->dlast ? p->dlast[at_bdn(p, b, d, n)] : 0.0;", "s->lam[n] = 0.0;", 0),
    ("bwd: dh0 without the first decay", "dh0[n] = L > 0 ? s->a[n] * s->lam[n] : s->lam[n];", "dh0[n] = s->lam[n];", 0),
    ("bwd: dh0 with the last decay", "dh0[n] = L > 0 ? s->a[n] * s->lam[n]", "dh0[n] = L > 0 ? s->a[(L - 1) * N + n] * s->lam[n]", 0),
    ("bwd: row list ignored", "int64_t r = row_id(j, i), b = r / p->Dch, d = r % p->Dch;\n            bwd_row",
     "int64_t r = i, b = r / p->Dch, d = r % p->Dch;\n            bwd_row", 0),
]

# Mistakes in the oracle's Python layer (the A_log map and its chain rule):
# (label, module attribute, replacement)
PY_MUTANTS = [
    ("A_log: sign", "a_from_log", lambda A_log: np.exp(np.asarray(A_log, np.float64))),
    ("A_log: exp dropped", "a_from_log", lambda A_log: -np.asarray(A_log, np.float64)),
    ("dA_log: chain rule dropped", "dA_log_rows", lambda dA_rows, A_rows: dA_rows),
    ("dA_log: divided by A", "dA_log_rows", lambda dA_rows, A_rows: dA_rows / A_rows),
]


def _apply(src, old, new, occ):
    idx = -1
    for _ in range(occ + 1):
        idx = src.find(old, idx + 1)
        assert idx >= 0, f"mutation anchor not found: {old!r}"
    return src[:idx] + new + src[idx + len(old):]


@pytest.mark.parametrize("label,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, label, old, new, occ):
    src = open(oracle.SRC).read()
    mutated = _apply(src, old, new, occ)
    assert mutated != src
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.build(src=path, out=os.path.join(tmp_path, "libmutant.so"), extra=("-DMUTANT",))
    orc = oracle.Oracle(lib)
    caught = []
    for check in P.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, RuntimeError, FloatingPointError) as e:  # noqa: PERF203
            caught.append((check.__name__, str(e)[:80]))
    assert caught, f"no pin caught mutant: {label}"


def _caught(orc):
    caught = []
    for check in P.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, RuntimeError, FloatingPointError) as e:  # noqa: PERF203
            caught.append((check.__name__, str(e)[:80]))
    return caught


@pytest.mark.parametrize("label,name,fn", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_pins_catch_python_mutant(monkeypatch, label, name, fn):
    monkeypatch.setattr(oracle, name, fn)
    assert _caught(oracle.Oracle()), f"no pin caught mutant: {label}"
