"""GPU parity of the token-wise layer stack (fw_decode_stack_step: per layer
the tcgen05 projections, the decode step, the output map, LayerNorm and the
feed-forward block, then the final norm) against the fp64 oracle
(oracle.stack.stack_step) on the same seeded weights and tokens, through the
C ABI.  Several tokens are stepped so the fast weights carry over between
calls.  Tolerance: max normwise relative error 2e-2 on the outputs and on
every layer's fast weights (bf16 operands, fp32 state and residual
stream)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import stack as ostack
from delta_rule_linear_dpfp_gb300 import binding as fw
from delta_rule_linear_dpfp_gb300 import build, inputs
from tests.parity_util import TOL_BF16, f64, maxrel

pytestmark = pytest.mark.gpu

NT = oracle.default_threads()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    fw.load()
    yield
    assert fw.fw_device_status() == fw.FW_OK


def _dev_layers(layers):
    return [{n: (None if t is None else t.cuda()) for n, t in ly.items()} for ly in layers]


def _np_layers(layers):
    return [{n: (None if t is None else f64(t)) for n, t in ly.items()} for ly in layers]


def _run(cfg, steps, w0_var=None, ldw_pad=0, seed=0, drop=()):
    B, H, d_key, nu, d_v, d_model, d_ff, nl = (cfg[n] for n in ("B", "H", "d_key", "nu", "d_v", "d_model",
                                                                  "d_ff", "n_layers"))
    d = inputs.stack_inputs(B, H, d_key, nu, d_v, d_model, d_ff, nl, steps, w0_var=w0_var, ldw_pad=ldw_pad,
                            seed=seed)
    for ly in d["layers"]:
        for n in drop:
            ly[n] = None
    dl = _dev_layers(d["layers"])
    ol = _np_layers(d["layers"])
    g, b = d["ln_gamma"].cuda(), d["ln_beta"].cuda()
    errs = []
    for t in range(steps):
        out = fw.fw_decode_stack_step(d["x"][t].cuda(), dl, H, d_key, d_v, nu=nu, ln_gamma=g, ln_beta=b)
        torch.cuda.synchronize()
        ref, _, states = ostack.stack_step(f64(d["x"][t]), ol, H, d_key, d_v, nu, f64(d["ln_gamma"]),
                                           f64(d["ln_beta"]), nthreads=NT)
        for ly, W in zip(ol, states):
            ly["W"] = W
        errs.append(maxrel(f64(out), ref))
    errs += [maxrel(f64(ly["W"]), o["W"]) for ly, o in zip(dl, ol)]
    return errs


SMALL = [  # B, H, d_key, nu, d_v, d_model, d_ff, n_layers
    (5, 2, 16, 2, 32, 128, 192, 3),      # a ragged row tile (5 of 128 rows), d_dot 64
    (130, 4, 32, 1, 16, 256, 320, 2),    # two row tiles, the second ragged; d_ff not a multiple of 128
    (3, 1, 64, 3, 64, 128, 64, 1),       # nu 3 (d_dot 384)
    # The cases above fold the LayerNorm into the first feed-forward map.  Below, a CTA of that map
    # would hold 4 K steps of 64 (more than its ring leaves room for beside the fp32 rows of x), so
    # the norm runs as its own kernel between the output map and the feed-forward block:
    (640, 2, 32, 1, 64, 256, 2048, 1),   # 80 output tiles: K not split
    (256, 4, 64, 1, 64, 1024, 2432, 1),  # d_model 1024, 38 output tiles: K in 4 slices of 4 steps
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "b{}h{}dk{}nu{}dv{}dm{}ff{}l{}".format(*c))
def test_stack_parity(case):
    cfg = dict(zip(("B", "H", "d_key", "nu", "d_v", "d_model", "d_ff", "n_layers"), case))
    errs = _run(cfg, steps=3, w0_var=0.01, ldw_pad=8, seed=sum(case))
    assert max(errs) <= TOL_BF16, errs


def test_stack_parity_full_size():
    # the benchmarked shape: 6 layers of d_model 512, 8 heads of 64, d_ff 2048, 256 sequences
    cfg = inputs.STACK_CONFIGS["stack_b256_l6"]
    errs = _run(cfg, steps=2, seed=3)
    assert max(errs) <= TOL_BF16, errs


def test_stack_without_biases_and_norm_parameters():
    cfg = dict(B=4, H=2, d_key=16, nu=1, d_v=32, d_model=128, d_ff=128, n_layers=2)
    errs = _run(cfg, steps=2, seed=5, drop=("b_o", "b_1", "b_2", "ln_gamma", "ln_beta"))
    assert max(errs) <= TOL_BF16, errs


def test_stack_zero_layers_is_the_final_norm():
    x = torch.randn(9, 256, generator=torch.Generator().manual_seed(1))
    g = torch.rand(256, generator=torch.Generator().manual_seed(2)) + 0.5
    out = fw.fw_decode_stack_step(x.cuda(), [], 4, 16, 16, ln_gamma=g.cuda())
    torch.cuda.synchronize()
    ref = ostack.layer_norm(f64(x), f64(g), None, 1e-5)
    assert maxrel(f64(out), ref) <= 1e-5


def test_stack_empty_batch_and_bad_arguments():
    cfg = dict(B=2, H=2, d_key=16, nu=1, d_v=32, d_model=128, d_ff=128, n_layers=1)
    d = inputs.stack_inputs(cfg["B"], cfg["H"], cfg["d_key"], cfg["nu"], cfg["d_v"], cfg["d_model"], cfg["d_ff"],
                            1, 1)
    dl = _dev_layers(d["layers"])
    empty = torch.empty(0, 128, device="cuda")
    assert fw.fw_decode_stack_step(empty, [dict(dl[0], W=torch.empty(0, 2, 32, 32, device="cuda"))], 2, 16,
                                   32).shape == (0, 128)
    with pytest.raises(fw.FwError):   # d_model not a multiple of 128
        fw.fw_decode_stack_step(torch.zeros(2, 64, device="cuda"), [], 2, 16, 32)
    assert fw.fw_decode_stack_workspace_size(2, 2, 16, 32, 96, 128) == 0
    assert fw.fw_decode_stack_workspace_size(2, 2, 16, 32, 128, 100) == 0


def test_stack_graph_replay_matches_eager():
    # one token step captured as a CUDA graph and replayed equals the eager call
    cfg = dict(B=8, H=2, d_key=32, nu=1, d_v=32, d_model=128, d_ff=256, n_layers=2)
    d = inputs.stack_inputs(cfg["B"], cfg["H"], cfg["d_key"], cfg["nu"], cfg["d_v"], cfg["d_model"], cfg["d_ff"],
                            cfg["n_layers"], 3, seed=11)
    d1, d2 = _dev_layers(d["layers"]), _dev_layers(d["layers"])
    xs = d["x"].cuda()
    ws = torch.empty(fw.fw_decode_stack_workspace_size(8, 2, 32, 32, 128, 256), dtype=torch.uint8, device="cuda")
    xin = xs[0].clone()
    out = torch.empty(8, 128, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fw.fw_decode_stack_step(xin, d2, 2, 32, 32, out=out, workspace=ws, stream=s)  # warm-up = token 0
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fw.fw_decode_stack_step(xin, d2, 2, 32, 32, out=out, workspace=ws, stream=s)
    for t in range(3):
        ref = fw.fw_decode_stack_step(xs[t], d1, 2, 32, 32)
        if t > 0:
            xin.copy_(xs[t])
            graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(ref, out), t
    for a, b in zip(d1, d2):
        assert torch.equal(a["W"], b["W"])
    assert np.isfinite(f64(out)).all()
