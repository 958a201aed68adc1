"""fp64 oracle of the token-wise layer stack.  TEST INFRASTRUCTURE ONLY.

Follows the Fast Weights Transformer guide (xdnf.cn/news/308600):
  - section "token_wise variant": the model keeps one fast-weight entry per
    layer, passes each token through every layer in turn, and applies the
    final LayerNorm to the result;
  - section "layer and model assembly": a layer adds the attention's output
    to its input (no norm before the attention), normalises the sum with
    its LayerNorm, and adds the feed-forward block's output; the block is
    linear (with bias), ReLU, linear (with bias); dropout is the identity at
    inference;
  - section "module structure": q, k, v and beta come from bias-free linear
    maps (beta through the sigmoid), and the heads' concatenated output goes
    through a linear layer with bias;
  - the fast-weight step itself is fw_oracle.c's decode step (the update
    rule of section "FastWeightsAttention: the new update rule").

LayerNorm is written out here (mean, biased variance, eps inside the square
root, then the elementwise gamma and beta) as PyTorch's LayerNorm defines
it.  Every array is numpy float64.
"""
import numpy as np

from . import delta_decode_step, project


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def layer_norm(x, gamma=None, beta=None, eps: float = 1e-5):
    """Normalise each row of x over its last axis: (x - mean) / sqrt(var +
    eps) with the biased variance, times gamma plus beta (one / zero when
    None)."""
    x = _f64(x)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    out = (x - mean) / np.sqrt(var + eps)
    if gamma is not None:
        out = out * _f64(gamma)
    if beta is not None:
        out = out + _f64(beta)
    return out


def _bias(b):
    return 0.0 if b is None else _f64(b)


def stack_step(x, layers, H: int, d_key: int, d_v: int, nu: int = 1, ln_gamma=None, ln_beta=None,
               eps: float = 1e-6, ln_eps: float = 1e-5, nthreads: int = 1):
    """One token of B sequences through the stack.

    x: [B, d_model]; layers: sequence of dicts with W_in [d_model, >= N]
    (N = H (2 d_key + d_v + 1); [W_q | W_k | W_v | W_beta] in its first N
    columns), W_o [H d_v, d_model], b_o, ln_gamma, ln_beta [d_model], W_1
    [d_model, d_ff], b_1 [d_ff], W_2 [d_ff, d_model], b_2 [d_model] (biases
    and norm parameters may be None) and W [B, H, d_v, d_dot], the layer's
    fast weights before this token.  Returns (out [B, d_model], the residual
    stream after the last layer [B, d_model], the list of the layers' fast
    weights after this token); nothing passed in is modified."""
    x = _f64(x)
    B, d_model = x.shape
    new_states = []
    for ly in layers:
        q, k, v, beta = project(x[:, None, :], ly["W_in"], H, d_key, d_v)   # [B, H, 1, *]
        y, W = delta_decode_step(q[:, :, 0], k[:, :, 0], v[:, :, 0], beta[:, :, 0], ly["W"], nu, eps,
                                 nthreads)
        new_states.append(W)
        x = x + y.reshape(B, H * d_v) @ _f64(ly["W_o"]) + _bias(ly.get("b_o"))
        z = layer_norm(x, ly.get("ln_gamma"), ly.get("ln_beta"), ln_eps)
        hidden = np.maximum(z @ _f64(ly["W_1"]) + _bias(ly.get("b_1")), 0.0)
        x = x + hidden @ _f64(ly["W_2"]) + _bias(ly.get("b_2"))
    return layer_norm(x, ln_gamma, ln_beta, ln_eps), x, new_states
