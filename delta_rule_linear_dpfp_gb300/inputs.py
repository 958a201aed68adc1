"""Seeded synthetic inputs for the fast-weight layer core.

This module only draws numbers: it holds none of the layer's arithmetic, so
both the CUDA path and the CPU oracle can take their inputs from it.  Every
tensor is drawn in fp32 from a CPU ``torch.Generator`` seeded with ``seed``,
in a fixed order, then rounded once to the I/O dtype; the same rounded bytes
feed the GPU and the oracle.

Workloads (shapes follow the Fast Weights Transformer guide's model: d_model
512, 8 heads of 64, nu = 1, and the chunked library's chunk of 64; the
guide's Tiny Shakespeare corpus is not used -- these synthetic tensors stand
in for its activations):

  tiny_f32        B1 H1 L64 d_key16 nu1 d_v16, fp32, chunk = L
  b4h8_l512       B4 H8 L512 d_key64 nu1 d_v64, bf16, chunk 64
  b2h8_l2048_nu3  B2 H8 L2048 d_key64 nu3 d_v64, bf16, chunk 64, W0 ~ N(0, 0.01)
  proj_d512       B1 H8 L1024 from x [1,1024,512] through bias-free random
                  projections W_q/W_k/W_v/W_beta ~ N(0, 1/512), bf16, chunk 64
  decode_b256     B256 H16 d_key64 nu2 d_v128, 128 tokens, bf16, W fp32 zeros
  stack_b256_l6   the guide's model shape for token-wise inference: 6 layers of
                  d_model 512, 8 heads of 64, nu 1, d_ff 2048; B256 sequences,
                  one token per step, every layer's W fp32 starting at zero

q, k, v ~ N(0, 1); beta = sigmoid(N(0, 1)); variances are the second
argument of N(.,.) (so W0 has standard deviation 0.1).
"""
import math

import torch

FORWARD_CONFIGS = {
    "tiny_f32": dict(B=1, H=1, L=64, d_key=16, nu=1, d_v=16, chunk=64, io="f32", w0_var=None),
    "b4h8_l512": dict(B=4, H=8, L=512, d_key=64, nu=1, d_v=64, chunk=64, io="bf16", w0_var=None),
    "b2h8_l2048_nu3": dict(B=2, H=8, L=2048, d_key=64, nu=3, d_v=64, chunk=64, io="bf16",
                           w0_var=0.01),
    # the same shape with 8x the batch (128 independent (b,h) sequences)
    "b16h8_l2048_nu3": dict(B=16, H=8, L=2048, d_key=64, nu=3, d_v=64, chunk=64, io="bf16",
                            w0_var=0.01),
    "proj_d512": dict(B=1, H=8, L=1024, d_key=64, nu=1, d_v=64, chunk=64, io="bf16", w0_var=None,
                      d_model=512),
}

DECODE_CONFIGS = {
    "decode_b256": dict(B=256, H=16, d_key=64, nu=2, d_v=128, steps=128, io="bf16", w0_var=None),
}

STACK_CONFIGS = {
    "stack_b256_l6": dict(B=256, H=8, d_key=64, nu=1, d_v=64, d_model=512, d_ff=2048, n_layers=6),
}

EPS = 1e-6


def torch_dtype(io: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def random_forward_inputs(B, H, L, d_key, nu, d_v, io="bf16", w0_var=None, seed=0):
    """q, k, v ~ N(0,1); beta = sigmoid(N(0,1)); optional W0 ~ N(0, w0_var).

    Draw order: q, k, v, beta logits, W0.  Returns a dict of CPU tensors:
    q, k [B,H,L,d_key], v [B,H,L,d_v], beta [B,H,L] in the I/O dtype, W0
    [B,H,d_v,2*d_key*nu] fp32 or None.
    """
    g = _gen(seed)
    dt = torch_dtype(io)
    q = torch.randn(B, H, L, d_key, generator=g, dtype=torch.float32)
    k = torch.randn(B, H, L, d_key, generator=g, dtype=torch.float32)
    v = torch.randn(B, H, L, d_v, generator=g, dtype=torch.float32)
    logits = torch.randn(B, H, L, generator=g, dtype=torch.float32)
    beta = torch.sigmoid(logits)
    W0 = None
    if w0_var is not None:
        W0 = torch.randn(B, H, d_v, 2 * d_key * nu, generator=g, dtype=torch.float32)
        W0 = W0 * math.sqrt(w0_var)
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                beta=beta.to(dt).contiguous(), W0=W0)


def linear_inputs(B, H, L, d_key, nu, d_v, with_state=False, seed=0):
    """Inputs of the sum rule (linear attention): q, k, v ~ N(0,1) in bf16;
    with_state adds W0 ~ N(0, 0.01) and a normaliser z0 = 0.05 |N(0,1)|
    (non-negative, like a running sum of DPFP features), both fp32.

    Draw order: q, k, v, W0, z0.  Returns a dict of CPU tensors.
    """
    g = _gen(seed)
    d_dot = 2 * d_key * nu
    q = torch.randn(B, H, L, d_key, generator=g, dtype=torch.float32)
    k = torch.randn(B, H, L, d_key, generator=g, dtype=torch.float32)
    v = torch.randn(B, H, L, d_v, generator=g, dtype=torch.float32)
    W0 = z0 = None
    if with_state:
        W0 = torch.randn(B, H, d_v, d_dot, generator=g, dtype=torch.float32) * 0.1
        z0 = torch.randn(B, H, d_dot, generator=g, dtype=torch.float32).abs() * 0.05
    bf = torch.bfloat16
    return dict(q=q.to(bf).contiguous(), k=k.to(bf).contiguous(), v=v.to(bf).contiguous(), W0=W0, z0=z0)


def projected_inputs(B, H, L, d_model, nu, io="bf16", seed=0):
    """x ~ N(0,1) [B,L,d_model] through bias-free W_q, W_k, W_v [d_model, d_model]
    and W_beta [d_model, H], all ~ N(0, 1/d_model), computed on the host in
    fp32 and rounded once; beta = sigmoid(x W_beta).  Heads split the
    projected features into H groups of d_model // H, laid out [B,H,L,d].
    Draw order: x, W_q, W_k, W_v, W_beta."""
    g = _gen(seed)
    dt = torch_dtype(io)
    d = d_model // H
    std = 1.0 / math.sqrt(d_model)
    x = torch.randn(B, L, d_model, generator=g, dtype=torch.float32)
    Wq = torch.randn(d_model, d_model, generator=g, dtype=torch.float32) * std
    Wk = torch.randn(d_model, d_model, generator=g, dtype=torch.float32) * std
    Wv = torch.randn(d_model, d_model, generator=g, dtype=torch.float32) * std
    Wb = torch.randn(d_model, H, generator=g, dtype=torch.float32) * std

    def heads(t):
        return t.reshape(B, L, H, d).permute(0, 2, 1, 3).contiguous()

    q, k, v = heads(x @ Wq), heads(x @ Wk), heads(x @ Wv)
    beta = torch.sigmoid(x @ Wb).permute(0, 2, 1).contiguous()
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                beta=beta.to(dt).contiguous(), W0=None)


def layer_inputs(B, H, L, d_model, d_key, d_v, nu=1, w0_var=None, seed=0):
    """Token activations and the four projection matrices side by side, for
    the forward from x: x ~ N(0,1) [B,L,d_model]; W_all = [W_q | W_k | W_v |
    W_beta] ~ N(0, 1/d_model) with H*d_key, H*d_key, H*d_v and H columns,
    padded with zero columns to a multiple of 8 (ldw); both rounded once to
    bf16.  Optional W0 ~ N(0, w0_var) fp32.  Draw order: x, W_all, W0."""
    g = _gen(seed)
    N = H * (2 * d_key + d_v + 1)
    ldw = (N + 7) // 8 * 8
    x = torch.randn(B, L, d_model, generator=g, dtype=torch.float32)
    W = torch.zeros(d_model, ldw, dtype=torch.float32)
    W[:, :N] = torch.randn(d_model, N, generator=g, dtype=torch.float32) / math.sqrt(d_model)
    W0 = None
    if w0_var is not None:
        W0 = torch.randn(B, H, d_v, 2 * d_key * nu, generator=g, dtype=torch.float32) * math.sqrt(w0_var)
    return dict(x=x.to(torch.bfloat16).contiguous(), W_all=W.to(torch.bfloat16).contiguous(), ldw=ldw, W0=W0)


def forward_inputs(name: str, seed: int = 0):
    cfg = FORWARD_CONFIGS[name]
    if "d_model" in cfg:
        return projected_inputs(cfg["B"], cfg["H"], cfg["L"], cfg["d_model"], cfg["nu"],
                                cfg["io"], seed)
    return random_forward_inputs(cfg["B"], cfg["H"], cfg["L"], cfg["d_key"], cfg["nu"],
                                 cfg["d_v"], cfg["io"], cfg["w0_var"], seed)


def decode_inputs(B, H, d_key, nu, d_v, steps, io="bf16", w0_var=None, seed=0):
    """Per-token inputs for `steps` decode steps: q, k [steps,B,H,d_key],
    v [steps,B,H,d_v], beta [steps,B,H] in the I/O dtype, and the initial
    persistent state W0 [B,H,d_v,2*d_key*nu] fp32 (zeros unless w0_var).
    Draw order: q, k, v, beta logits, W0."""
    g = _gen(seed)
    dt = torch_dtype(io)
    q = torch.randn(steps, B, H, d_key, generator=g, dtype=torch.float32)
    k = torch.randn(steps, B, H, d_key, generator=g, dtype=torch.float32)
    v = torch.randn(steps, B, H, d_v, generator=g, dtype=torch.float32)
    beta = torch.sigmoid(torch.randn(steps, B, H, generator=g, dtype=torch.float32))
    if w0_var is None:
        W0 = torch.zeros(B, H, d_v, 2 * d_key * nu, dtype=torch.float32)
    else:
        W0 = torch.randn(B, H, d_v, 2 * d_key * nu, generator=g, dtype=torch.float32)
        W0 = W0 * math.sqrt(w0_var)
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                beta=beta.to(dt).contiguous(), W0=W0)


def stack_inputs(B, H, d_key, nu, d_v, d_model, d_ff, n_layers, steps, w0_var=None, ldw_pad=0, seed=0):
    """Random-init weights of an n_layers token-wise stack and `steps` tokens.

    x ~ N(0,1) [steps, B, d_model] fp32.  Per layer: W_in = [W_q | W_k | W_v |
    W_beta] ~ N(0, 1/d_model) ([d_model, ldw], ldw = N rounded up to 8 plus
    ldw_pad zero columns), W_o ~ N(0, 1/(H d_v)), W_1 ~ N(0, 1/d_model), W_2 ~
    N(0, 1/d_ff) (bf16, [in, out]); b_o, b_1, b_2 ~ N(0, 0.01); ln_gamma = 1 +
    N(0, 0.01), ln_beta ~ N(0, 0.01) (fp32); the layer's fast weights W fp32
    [B, H, d_v, 2 d_key nu], zeros unless w0_var.  Then the final norm's
    gamma and beta as above.  Draw order: x, then each layer's W_in, W_o,
    b_o, ln_gamma, ln_beta, W_1, b_1, W_2, b_2, W, then the final gamma,
    beta."""
    g = _gen(seed)
    N = H * (2 * d_key + d_v + 1)
    ldw = (N + 7) // 8 * 8 + ldw_pad

    def rn(*shape, std=1.0):
        return torch.randn(*shape, generator=g, dtype=torch.float32) * std

    x = rn(steps, B, d_model)
    layers = []
    for _ in range(n_layers):
        W_in = torch.zeros(d_model, ldw, dtype=torch.float32)
        W_in[:, :N] = rn(d_model, N, std=1.0 / math.sqrt(d_model))
        ly = dict(W_in=W_in.to(torch.bfloat16).contiguous(),
                  W_o=rn(H * d_v, d_model, std=1.0 / math.sqrt(H * d_v)).to(torch.bfloat16).contiguous(),
                  b_o=rn(d_model, std=0.1), ln_gamma=1.0 + rn(d_model, std=0.1), ln_beta=rn(d_model, std=0.1),
                  W_1=rn(d_model, d_ff, std=1.0 / math.sqrt(d_model)).to(torch.bfloat16).contiguous(),
                  b_1=rn(d_ff, std=0.1),
                  W_2=rn(d_ff, d_model, std=1.0 / math.sqrt(d_ff)).to(torch.bfloat16).contiguous(),
                  b_2=rn(d_model, std=0.1))
        d_dot = 2 * d_key * nu
        ly["W"] = (torch.zeros(B, H, d_v, d_dot, dtype=torch.float32) if w0_var is None
                   else rn(B, H, d_v, d_dot, std=math.sqrt(w0_var)))
        layers.append(ly)
    return dict(x=x, layers=layers, ln_gamma=1.0 + rn(d_model, std=0.1), ln_beta=rn(d_model, std=0.1))
