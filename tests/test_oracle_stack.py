"""Pins of the token-wise layer stack oracle (oracle/stack.py), and planted
mistakes in a copy of it that those pins must catch (CPU only)."""
import os
import types

import pytest

import oracle
from oracle import stack
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.abspath(stack.__file__)), "stack.py")


@pytest.mark.parametrize("pin", oracle_pins.STACK_PINS, ids=lambda p: p.__name__)
def test_stack_pin(pin):
    pin(oracle.lib(), stack)


MUTANTS = {
    "attention_residual_dropped": ('x = x + y.reshape(B, H * d_v) @ _f64(ly["W_o"])',
                                   'x = y.reshape(B, H * d_v) @ _f64(ly["W_o"])'),
    "output_bias_dropped": (' + _bias(ly.get("b_o"))', ''),
    "heads_concatenated_value_major": ('y.reshape(B, H * d_v)', 'y.transpose(0, 2, 1).reshape(B, H * d_v)'),
    "feed_forward_reads_unnormalised": ('hidden = np.maximum(z @', 'hidden = np.maximum(x @'),
    "relu_dropped": ('hidden = np.maximum(z @ _f64(ly["W_1"]) + _bias(ly.get("b_1")), 0.0)',
                     'hidden = z @ _f64(ly["W_1"]) + _bias(ly.get("b_1"))'),
    "feed_forward_residual_dropped": ('x = x + hidden @', 'x = hidden @'),
    "norm_unbiased_variance": ('var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)',
                               'var = ((x - mean) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)'),
    "norm_eps_outside_root": ('np.sqrt(var + eps)', '(np.sqrt(var) + eps)'),
    "norm_beta_dropped": ('        out = out + _f64(beta)\n', '        out = out + 0.0\n'),
    "state_not_carried": ('new_states.append(W)', 'new_states.append(_f64(ly["W"]))'),
    "final_norm_dropped": ('return layer_norm(x, ln_gamma, ln_beta, ln_eps), x, new_states',
                           'return x, x, new_states'),
    "norm_before_attention": ('q, k, v, beta = project(x[:, None, :]',
                              'q, k, v, beta = project(layer_norm(x, None, None, ln_eps)[:, None, :]'),
    "norm_gamma_dropped": ('        out = out * _f64(gamma)\n', '        out = out * 1.0\n'),
    "norm_mean_not_subtracted": ('out = (x - mean) / np.sqrt(var + eps)', 'out = x / np.sqrt(var + eps)'),
    "norm_parameters_swapped": ('layer_norm(x, ly.get("ln_gamma"), ly.get("ln_beta"), ln_eps)',
                                'layer_norm(x, ly.get("ln_beta"), ly.get("ln_gamma"), ln_eps)'),
    "hidden_bias_dropped": (' + _bias(ly.get("b_1"))', ''),
    "second_feed_forward_bias_dropped": (' + _bias(ly.get("b_2"))', ''),
}


def _mutant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, name
    mod = types.ModuleType("oracle._stack_" + name)
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), SRC + ":" + name, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_stack_mutant_is_caught(name):
    mod = _mutant(name, *MUTANTS[name])
    failed = []
    for pin in oracle_pins.STACK_PINS:
        try:
            pin(oracle.lib(), mod)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no stack pin notices the mutation {name}"
