"""Planted mistakes in the oracle must fail its pins (CPU only).

Each case copies oracle/fw_oracle.c to a temporary folder, applies one textual
mutation of the kind a plausible slip would make (a wrong roll direction, a
dropped term, a wrong sign, a swapped operand, the read taken before the
write, ...), compiles it, and runs every pin from tests/oracle_pins.py against
it.  At least one pin has to fail, otherwise the pins would not notice that
mistake in the oracle.
"""
import os
import subprocess

import pytest

from oracle import OracleLib
from oracle.build import SRC
from oracle.chunked import delta_backward_chunked, delta_forward_chunked
from tests import oracle_pins

MUTANTS = {
    "roll_direction": ("int src = ((j - i) % n + n) % n;", "int src = ((j + i) % n + n) % n;"),
    "relu_of_minus_k_dropped": ("x[d_key + j] = -k[j] > 0.0 ? -k[j] : 0.0;",
                                "x[d_key + j] = k[j] > 0.0 ? k[j] : 0.0;"),
    "eps_dropped": ("phi[m] = phi[m] / (s + eps);", "phi[m] = phi[m] / (s);"),
    "not_normalised": ("phi[m] = phi[m] / (s + eps);", "phi[m] = phi[m] + 0.0 * eps;"),
    "retrieve_with_query": ("acc += W[(size_t)r * d_dot + m] * pk[m];\n            vbar[r] = acc;",
                            "acc += W[(size_t)r * d_dot + m] * pq[m];\n            vbar[r] = acc;"),
    "update_sign": ("W[(size_t)r * d_dot + m] += u * pk[m];", "W[(size_t)r * d_dot + m] -= u * pk[m];"),
    "beta_on_value_only": ("double u = beta[t] * (v[t * d_v + r] - vbar[r]);",
                           "double u = beta[t] * v[t * d_v + r] - vbar[r];"),
    "write_with_query": ("W[(size_t)r * d_dot + m] += u * pk[m];", "W[(size_t)r * d_dot + m] += u * pq[m];"),
    "read_before_write": ("acc += W[(size_t)r * d_dot + m] * pq[m];\n            y[t * d_v + r] = acc;",
                          "acc += (W[(size_t)r * d_dot + m] - beta[t] * (v[t * d_v + r] - vbar[r]) * pk[m])"
                          " * pq[m];\n            y[t * d_v + r] = acc;"),
    "initial_state_ignored": ("memcpy(W, j->W0 + bh * wsz, sizeof(double) * wsz);",
                              "memset(W, 0, sizeof(double) * wsz);"),
    "state_transposed": ("W[(size_t)r * d_dot + m] += u * pk[m];",
                         "W[(size_t)m * d_v + r] += u * pk[m];"),
    # the sum rule (linear attention)
    "sum_rule_writes_query": ("W[(size_t)r * d_dot + m] += v[t * d_v + r] * pk[m];",
                              "W[(size_t)r * d_dot + m] += v[t * d_v + r] * pq[m];"),
    "sum_rule_z_not_accumulated": ("z[m] += pk[m];", "z[m] = pk[m];"),
    "sum_rule_denominator_with_key": ("den += z[m] * pq[m];", "den += z[m] * pk[m];"),
    "sum_rule_read_before_write": ("        for (int m = 0; m < d_dot; ++m)\n            z[m] += pk[m];\n",
                                   "        for (int m = 0; m < d_dot; ++m)\n            z[m] += 0.0 * pk[m];\n"),
    "sum_rule_initial_z_ignored": ("z[m] = j->z0 ? j->z0[bh * d_dot + m] : 0.0;", "z[m] = 0.0;"),
    # the backward
    "backward_state_sign": ("gW[(size_t)r * d_dot + m] -= beta[t] * gu[r] * pkt[m];",
                            "gW[(size_t)r * d_dot + m] += beta[t] * gu[r] * pkt[m];"),
    "backward_key_drops_retrieve": ("acc += gW[(size_t)r * d_dot + m] * u - Wp[(size_t)r * d_dot + m] * beta[t] * gu[r];",
                                    "acc += gW[(size_t)r * d_dot + m] * u;"),
    "backward_query_with_old_state": ("acc += Wn[(size_t)r * d_dot + m] * gy[t * d_v + r];",
                                      "acc += Wp[(size_t)r * d_dot + m] * gy[t * d_v + r];"),
    "backward_normaliser_term_dropped": ("const double gp = gphi[m] / (s + eps) - gp_dot_p / ((s + eps) * (s + eps));",
                                         "const double gp = gphi[m] / (s + eps);"),
    "backward_roll_partner_dropped": ("            gx[src] += gp * x[j];\n", "\n"),
    "backward_roll_partner_wrong": ("gx[j] += gp * x[src];", "gx[j] += gp * x[j];"),
    "backward_beta_grad_drops_retrieve": ("gb += gu[r] * (v[t * d_v + r] - a[t * d_v + r]);",
                                          "gb += gu[r] * v[t * d_v + r];"),
    "backward_value_grad_drops_beta": ("gv[t * d_v + r] = beta[t] * gu[r];", "gv[t * d_v + r] = gu[r];"),
    "backward_readout_grad_with_key": ("gW[(size_t)r * d_dot + m] += gy[t * d_v + r] * pqt[m];",
                                       "gW[(size_t)r * d_dot + m] += gy[t * d_v + r] * pkt[m];"),
    "backward_final_state_grad_ignored": ("gW[e] = gWL ? gWL[e] : 0.0;", "gW[e] = 0.0;"),
    "backward_minus_k_branch_sign": ("gk[j] = (k[j] > 0.0 ? gx[j] : 0.0) - (-k[j] > 0.0 ? gx[d_key + j] : 0.0);",
                                     "gk[j] = (k[j] > 0.0 ? gx[j] : 0.0) + (-k[j] > 0.0 ? gx[d_key + j] : 0.0);"),
    "backward_key_grad_with_new_state": ("- Wp[(size_t)r * d_dot + m] * beta[t] * gu[r];",
                                         "- Wn[(size_t)r * d_dot + m] * beta[t] * gu[r];"),
    # the DPFP map: the shift off by one (block 1 = x * x), the normaliser over block 1 only
    "dpfp_shift_off_by_one": ("int src = ((j - i) % n + n) % n;", "int src = ((j - i + 1) % n + n) % n;"),
    "dpfp_sum_over_first_block": ("            s += p;\n", "            s += (i == 1) ? p : 0.0;\n"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found in the oracle"
    mutated = src.replace(old, new, 1)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o",
                    str(so), str(c), "-lpthread", "-lm"], check=True)
    return OracleLib(str(so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    o = _build_mutant(tmp_path, name, old, new)
    failed = []
    pins = list(oracle_pins.ALL_PINS) + [
        lambda ob: oracle_pins.pin_chunked_equals_sequential(ob, delta_forward_chunked),
        lambda ob: oracle_pins.pin_chunked_backward_equals_sequential(ob, delta_backward_chunked)]
    for pin in pins:
        try:
            pin(o)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(getattr(pin, "__name__", "chunked"))
    assert failed, f"no pin caught the planted mistake '{name}'"


# The projections (oracle.project, numpy): each mutant is the function's own
# source with one textual change, executed in the oracle module's namespace
# and put in its place for the projection pin.
PROJECTION_MUTANTS = {
    "beta_sigmoid_sign": ("np.exp(-P[", "np.exp(P["),
    "heads_split_feature_major": ("a.reshape(B, L, H, d).transpose(0, 2, 1, 3)",
                                  "a.reshape(B, L, d, H).transpose(0, 3, 1, 2)"),
    "query_and_key_swapped": ("q = heads(P[..., :nq], d_key)\n    k = heads(P[..., nq:2 * nq], d_key)",
                              "k = heads(P[..., :nq], d_key)\n    q = heads(P[..., nq:2 * nq], d_key)"),
    "value_from_the_key_block": ("v = heads(P[..., 2 * nq:2 * nq + nv], d_v)", "v = heads(P[..., nq:nq + nv], d_v)"),
    "beta_from_the_first_columns": ("P[..., 2 * nq + nv:2 * nq + nv + H]", "P[..., 0:H]"),
}


@pytest.mark.parametrize("name", sorted(PROJECTION_MUTANTS))
def test_projection_mutant_is_caught(monkeypatch, name):
    import inspect
    import textwrap

    import oracle
    old, new = PROJECTION_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(oracle.project))
    assert src.count(old) == 1, f"mutation anchor for {name} not found in oracle.project"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    monkeypatch.setattr(oracle, "project", ns["project"])
    with pytest.raises((AssertionError, ValueError, IndexError)):
        oracle_pins.pin_projection_selection(None)


def test_projection_copy_without_mutation_passes(monkeypatch):
    """The control for the cases above: the unchanged source, put in place the
    same way, passes the pin."""
    import inspect
    import textwrap

    import oracle
    ns = dict(vars(oracle))
    exec(compile(textwrap.dedent(inspect.getsource(oracle.project)), "<copy>", "exec"), ns)
    monkeypatch.setattr(oracle, "project", ns["project"])
    oracle_pins.pin_projection_selection(None)
