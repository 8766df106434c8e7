"""Post-expert RMSNorm ("Meta Dist-MoE: Open-Source Fused MoE Kernels for
Blackwell", "Supported modes"; reading: the layer's BF16 output row x is
normalised over D with a per-feature gamma, y = bf16(gamma x r),
r = 1/sqrt(mean x^2 + eps)) against the oracle (oracle/post_norm.py):

* the pre-norm rows a training forward saves are bit-identical to the
  output of the same layer without the norm (the norm reads what the layer
  would have written);
* the normalised output equals the oracle applied to those rows within one
  BF16 step per element (r and the products are FP32 on the GPU), and the
  whole forward agrees with the fp64 oracle within the precision's
  tolerance, also when accumulating onto a shared expert's output and for a
  token whose routes are all inactive;
* the backward (dx of the pre-norm rows, dgamma) agrees with the oracle on
  the same rows, and dgamma is bitwise reproducible;
* argument errors.
"""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import abi, synth
from oracle import post_norm as pn

from moe_cases import TOL, Case, rel_err, run_oracle, to_f64

pytestmark = pytest.mark.gpu

EPS = 1e-5


def _case(precision, seed):
    w = synth.Workload(f"norm_{precision}", 192, 256, 256, 8, 2, precision, "zipf", inactive_frac=0.05,
                       zipf_s=1.2, seed=seed)
    ids, s = synth.make_routing(w)
    ids[0, :] = -1          # a token with no active route
    s[0, :] = 0.0
    return Case(w, ids=ids, scores=s)


def _gamma(D, seed):
    g = np.random.default_rng(seed).normal(1.0, 0.25, size=D)
    return torch.from_numpy(g).to(torch.bfloat16).to("cuda")


def _run(case, precision, post_norm, gamma=None, training=True, out_init=None):
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    w = case.w
    dev = torch.device("cuda")
    layer = MoELayer(case.T, w.D, w.F, w.E, w.K, precision, training=training, post_norm=post_norm)
    if post_norm:
        layer.set_post_norm(gamma, EPS)
    W13 = PreparedWeight(case.w13.to(dev), precision, with_transpose=training)
    W2 = PreparedWeight(case.w2.to(dev), precision, with_transpose=training)
    out = torch.zeros((case.T, w.D), dtype=torch.bfloat16, device=dev)
    if out_init is not None:
        out.copy_(out_init)
    saved = layer.new_saved() if training else None
    layer.forward(case.x.to(dev), torch.from_numpy(case.ids).to(dev), torch.from_numpy(case.scores).to(dev), W13, W2,
                  out=out, saved=saved, accumulate=out_init is not None)
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    return layer, saved, out


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
@pytest.mark.parametrize("accumulate", [False, True])
def test_post_norm_forward(precision, accumulate):
    case = _case(precision, 61)
    D = case.w.D
    gamma = _gamma(D, 62)
    init = None
    if accumulate:
        init = torch.from_numpy(np.random.default_rng(63).normal(0.0, 0.05, (case.T, D))).to(torch.bfloat16).cuda()
    _, _, plain = _run(case, precision, False, out_init=init)
    layer, saved, y = _run(case, precision, True, gamma, out_init=init)
    x = layer.saved_field(saved, abi.MOE_SAVED_PRENORM, torch.bfloat16, (case.T, D))
    assert torch.equal(x, plain)
    g64 = to_f64(gamma)
    want, _ = pn.forward(to_f64(x), g64, EPS)
    got = to_f64(y)
    step = np.maximum(np.abs(want), 2.0 ** -126) * 2.0 ** -7      # one BF16 step
    assert np.all(np.abs(got - want) <= step)
    assert np.mean(got == want) > 0.99
    if init is None:
        assert np.all(got[0] == 0.0)          # a token with no active route stays exactly zero
    # the whole forward against the fp64 oracle
    o = run_oracle(case, out_init=None if init is None else to_f64(init), backward=False)
    want_full, _ = pn.forward(o["out"], g64, EPS)
    assert rel_err(got, want_full) <= TOL[precision]
    # inference: same output, nothing saved
    _, _, y_inf = _run(case, precision, True, gamma, training=False, out_init=init)
    assert torch.equal(y_inf, y)


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_post_norm_backward(precision):
    case = _case(precision, 64)
    D = case.w.D
    gamma = _gamma(D, 65)
    layer, saved, _ = _run(case, precision, True, gamma)
    x = to_f64(layer.saved_field(saved, abi.MOE_SAVED_PRENORM, torch.bfloat16, (case.T, D)))
    dy = torch.from_numpy(np.random.default_rng(66).normal(size=(case.T, D))).to(torch.bfloat16).cuda()
    dx, dg = layer.post_norm_backward(saved, dy)
    torch.cuda.synchronize()
    want_dx, want_dg = pn.backward(x, to_f64(gamma), EPS, to_f64(dy))
    assert rel_err(to_f64(dx), want_dx) <= 2.0 ** -7
    np.testing.assert_allclose(dg.cpu().numpy().astype(np.float64), want_dg, rtol=1e-4, atol=1e-4)
    _, dg2 = layer.post_norm_backward(saved, dy)
    assert torch.equal(dg, dg2)
    # the pre-norm gradient feeds the layer's own backward
    dxl, dW13, dW2 = layer.backward(saved, dx, *_weights(case, precision))
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    assert torch.isfinite(dxl.float()).all() and torch.isfinite(dW13.float()).all()


def _weights(case, precision):
    from mixture_experts_routed_route_gb300.layer import PreparedWeight
    dev = torch.device("cuda")
    return (PreparedWeight(case.w13.to(dev), precision, with_transpose=True),
            PreparedWeight(case.w2.to(dev), precision, with_transpose=True))


def test_post_norm_argument_errors():
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    case = _case("bf16", 67)
    w = case.w
    gamma = _gamma(w.D, 68)
    plain = MoELayer(case.T, w.D, w.F, w.E, w.K, "bf16")
    with pytest.raises(abi.MoEError):          # context without MOE_POST_NORM
        plain.set_post_norm(gamma, EPS)
    layer = MoELayer(case.T, w.D, w.F, w.E, w.K, "bf16", post_norm=True)
    for eps in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(abi.MoEError):
            layer.set_post_norm(gamma, eps)
    dev = torch.device("cuda")
    W13 = PreparedWeight(case.w13.to(dev), "bf16", with_transpose=False)
    W2 = PreparedWeight(case.w2.to(dev), "bf16", with_transpose=False)
    with pytest.raises(abi.MoEError) as ei:    # no gamma set yet
        layer.forward(case.x.to(dev), torch.from_numpy(case.ids).to(dev), torch.from_numpy(case.scores).to(dev),
                      W13, W2)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    layer.set_post_norm(gamma, EPS)
    out = layer.forward(case.x.to(dev), torch.from_numpy(case.ids).to(dev), torch.from_numpy(case.scores).to(dev),
                        W13, W2)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    with pytest.raises(abi.MoEError):          # backward needs a training context
        layer.post_norm_backward(layer.new_saved(), out)
    plain.close()
    layer.close()
