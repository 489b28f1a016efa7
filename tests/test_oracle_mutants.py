"""The oracle's pins reject plausible mistakes.

Each mutant is a copy of oracle/gn3d_oracle.c with one plausible mistake: a
dropped term, a wrong sign, index, divisor or rounding step. It is compiled
into a temporary library, and tests/test_oracle.py runs against it in a child
process (GN3D_ORACLE_LIB); every mutant must make a pin fail.  The
channels-last adapters are mutated in-process, with a transposed reshape or a
wrong index map, and their pins must fail too.  The real oracle source is
never modified.
"""
import os
import subprocess
import sys
import types

import numpy as np
import pytest

import oracle

from . import test_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gn3d_oracle.c")

MUTANTS = {
    "eps_outside_sqrt": ("rstd[ng] = 1.0 / sqrt(v + e);", "rstd[ng] = 1.0 / sqrt(v) + e;"),
    "unbiased_variance": ("const double v = M ? nsum_val(&s2) / (double)M : 0.0;",
                          "const double v = M > 1 ? nsum_val(&s2) / (double)(M - 1) : 0.0;"),
    "eps_not_fp32": ("static double eps_as_used(double eps) { return (double)(float)eps; }",
                     "static double eps_as_used(double eps) { return eps; }"),
    "beta_sign": ("return (xv - mu) * r * gam + bet;", "return (xv - mu) * r * gam - bet;"),
    "gamma_index": ("const double gam = param(gamma, c, 1.0), bet = param(beta, c, 0.0);",
                    "const double gam = param(gamma, c / Cg, 1.0), bet = param(beta, c, 0.0);"),
    "dx_drop_a": ("return r * (dyv * gam - a - xh * b);", "return r * (dyv * gam - xh * b);"),
    "dx_drop_b": ("return r * (dyv * gam - a - xh * b);", "return r * (dyv * gam - a);"),
    "dx_sign_b": ("return r * (dyv * gam - a - xh * b);", "return r * (dyv * gam - a + xh * b);"),
    "dgamma_without_xhat": ("nsum_add(&sdyx, d * xh);", "nsum_add(&sdyx, d);"),
    "b_without_gamma": ("nsum_add(&sgx, d * gam * xh);", "nsum_add(&sgx, d * xh);"),
    "bf16_widening": ("<< 16;", "<< 15;"),
    "bf16_rounding_position": ("int q = e - 8;", "int q = e - 9;"),
    "group_base": ("const int64_t base = ng * M;", "const int64_t base = ng * S;"),
    "relu_minus_zero": ("out[i] = (v[i] < 0.0) ? 0.0 : v[i];", "out[i] = (v[i] <= 0.0) ? 0.0 : v[i];"),
    "relu_gate_strict": ("if (gate && widen(gate, dtype, i) <= 0.0) return 0.0;",
                         "if (gate && widen(gate, dtype, i) < 0.0) return 0.0;"),
    "relu_at_gated_by_x": ("return backward_at_impl(dy, out, x, dtype,", "return backward_at_impl(dy, x, x, dtype,"),
    "sums_rows_swapped": ("if (s1) memcpy(s1, db, sizeof(double) * (size_t)NC);",
                          "if (s1) memcpy(s1, dg, sizeof(double) * (size_t)NC);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    a, b = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(a) == 1, f"mutation anchor for {name} not found once"
    msrc = tmp_path / "gn3d_oracle.c"
    msrc.write_text(src.replace(a, b))
    lib = oracle.compile_source(str(msrc), str(tmp_path / "libgn3d_oracle_mutant.so"))
    env = dict(os.environ, GN3D_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle.py", "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-1500:]}"
    assert " failed" in r.stdout, f"mutant {name} did not fail a pin (collection or build error?):\n{r.stdout[-1500:]}"


def _mutated_oracle(**overrides):
    m = types.SimpleNamespace(**{k: getattr(oracle, k) for k in dir(oracle) if not k.startswith("__")})
    for k, v in overrides.items():
        setattr(m, k, v)
    return m


def _wrong_to_ncdhw(a, N, C, S):
    return np.ascontiguousarray(np.asarray(a).reshape(N, C, S)).reshape(-1)  # no transpose


def _wrong_to_ndhwc(a, N, C, S):
    return np.ascontiguousarray(np.asarray(a).reshape(N, S, C)).reshape(-1)  # no transpose


def _fwd_with(to_ncdhw, to_ndhwc):
    def forward_ndhwc(x, gamma, beta, N, C, S, G, eps):
        y, mean, rstd = oracle.forward(to_ncdhw(x, N, C, S), gamma, beta, N, C, S, G, eps)
        return to_ndhwc(y, N, C, S), mean, rstd
    return forward_ndhwc


def _bwd_with(to_ncdhw, to_ndhwc):
    def backward_ndhwc(dy, x, mean, rstd, gamma, N, C, S, G, want_dx=True):
        dx, dg, db = oracle.backward(to_ncdhw(dy, N, C, S), to_ncdhw(x, N, C, S), mean, rstd, gamma, N, C, S, G,
                                     want_dx)
        return (to_ndhwc(dx, N, C, S) if want_dx else None), dg, db
    return backward_ndhwc


def test_channels_last_pins_reject_mutants():
    mutants = {
        "untransposed_input": _mutated_oracle(forward_ndhwc=_fwd_with(_wrong_to_ncdhw, oracle.ncdhw_to_ndhwc),
                                              backward_ndhwc=_bwd_with(_wrong_to_ncdhw, oracle.ncdhw_to_ndhwc),
                                              ndhwc_to_ncdhw=_wrong_to_ncdhw),
        "untransposed_output": _mutated_oracle(forward_ndhwc=_fwd_with(oracle.ndhwc_to_ncdhw, _wrong_to_ndhwc),
                                               backward_ndhwc=_bwd_with(oracle.ndhwc_to_ncdhw, _wrong_to_ndhwc),
                                               ncdhw_to_ndhwc=_wrong_to_ndhwc),
        "index_map_swapped": _mutated_oracle(
            ndhwc_index=lambda idx, N, C, S: (np.asarray(idx) % S) * C + np.asarray(idx) // S),
    }
    pins = [test_oracle.test_ndhwc_layout_brute_force, test_oracle.test_ndhwc_matches_torch_channels_last_float64,
            test_oracle.test_ndhwc_index_and_permutations_agree]
    for name, orc in mutants.items():
        caught = False
        for pin in pins:
            try:
                pin(orc)
            except (AssertionError, ValueError, IndexError):
                caught = True
                break
        assert caught, f"channels-last mutant {name} survived the pins"


def _relu_ndhwc_gated_by_x(dy, x, out, mean, rstd, gamma, N, C, S, G, want_dx=True):
    return oracle.backward_relu_ndhwc(dy, x, x, mean, rstd, gamma, N, C, S, G, want_dx)  # x passed as the gate


def _combine_without_cross_term(parts):
    n, m, q = (np.array(v, dtype=np.float64) for v in parts[0])
    for nb, mb, qb in parts[1:]:
        tot = n + nb
        m = m + (mb - m) * nb / tot
        q = q + qb  # the d^2 * na * nb / n term dropped
        n = tot
    return n, m, q


def _combine_unweighted_mean(parts):
    n, m, q = (np.array(v, dtype=np.float64) for v in parts[0])
    for nb, mb, qb in parts[1:]:
        d = mb - m
        tot = n + nb
        q = q + qb + d * d * n * nb / tot
        m = (m + mb) / 2  # means averaged, not weighted by the counts
        n = tot
    return n, m, q


def test_relu_ndhwc_and_sharded_pins_reject_mutants():
    cases = {
        "relu_ndhwc_gated_by_x": (_mutated_oracle(backward_relu_ndhwc=_relu_ndhwc_gated_by_x),
                                  [test_oracle.test_backward_relu_ndhwc_matches_torch_channels_last]),
        "combine_without_cross_term": (
            _mutated_oracle(combine_moments=_combine_without_cross_term),
            [test_oracle.test_combine_moments_textbook,
             lambda o: test_oracle.test_sharded_moments_combine_to_the_whole(o, [1, 2, 1])]),
        "combine_unweighted_mean": (
            _mutated_oracle(combine_moments=_combine_unweighted_mean),
            [test_oracle.test_combine_moments_textbook,
             lambda o: test_oracle.test_sharded_moments_combine_to_the_whole(o, [3, 1])]),
    }
    for name, (orc, pins) in cases.items():
        caught = False
        for pin in pins:
            try:
                pin(orc)
            except (AssertionError, ValueError, IndexError):
                caught = True
                break
        assert caught, f"mutant {name} survived the pins"
