"""Layer variants of "Meta Dist-MoE: Open-Source Fused MoE Kernels for
Blackwell", "Supported modes", against the oracle:

* clamped SwiGLU (limit L: h2 = SiLU(min(g, L)) * clamp(u, -L, L), gradients
  masked outside the clamp range), forward and backward, BF16 and MXFP8;
* clip statistics: the device counts of clamped gate / up values equal the
  counts taken from the GPU's own saved BF16 h1 (the same decisions), and
  agree with the oracle's counts up to values within a BF16 step of L;
* 1x32 inference weights: codes and scales bit-exact, forward within the
  MXFP8 tolerance, and rejected by the backward.
"""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import abi, synth
from oracle import formats as fm

from moe_cases import (TOL, Case, check_mx_wgrad, rel_err, run_gpu, run_oracle, to_f64, unpack_weight_sf)

pytestmark = pytest.mark.gpu

LIMIT = 1.0     # h1 ~ N(0, 1) at these shapes: about 16 % of g and 32 % of u clip


def _case(precision, seed):
    w = synth.Workload(f"clamp_{precision}", 200, 256, 256, 8, 2, precision, "zipf", inactive_frac=0.05,
                       zipf_s=1.2, seed=seed)
    return Case(w)


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_clamped_swiglu_forward_backward(precision):
    case = _case(precision, 41 if precision == "bf16" else 42)
    g = run_gpu(case, swiglu_limit=LIMIT)
    o = run_oracle(case, swiglu_limit=LIMIT)
    assert g["err_bits"] == 0
    st = o["state"]
    Fh = st["F"]
    h1 = st["h1"]
    assert np.mean(h1[:, :Fh] > LIMIT) > 0.05 and np.mean(np.abs(h1[:, Fh:]) > LIMIT) > 0.05   # clamp active
    for k in ("out", "dx", "dp"):
        assert rel_err(g[k], o[k]) <= TOL[precision], k
    if precision == "mxfp8":
        check_mx_wgrad(g["dW13"], g["dW2"], st, o["grads"])
    else:
        assert rel_err(g["dW13"], o["dW13"]) <= TOL[precision]
        assert rel_err(g["dW2"], o["dW2"]) <= TOL[precision]
    # the clamp changes the result: the plain SwiGLU oracle is measurably off
    plain = run_oracle(case, backward=False)
    assert rel_err(plain["out"], o["out"]) > 3 * TOL[precision]


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_clip_statistics(precision):
    case = _case(precision, 43)
    g = run_gpu(case, swiglu_limit=LIMIT, backward=False)
    layer, saved = g["layer"], g["saved"]
    F = case.w.F
    hdr = layer.saved_field(saved, abi.MOE_SAVED_HEADER, torch.int32, (16,)).cpu().numpy()
    rows = int(hdr[2])
    h1 = to_f64(layer.saved_field(saved, abi.MOE_SAVED_H1, torch.bfloat16, (layer.r_cap, 2 * F))[:rows])
    want = (int(np.sum(h1[:, :F] > LIMIT)), int(np.sum(np.abs(h1[:, F:]) > LIMIT)))
    got = layer.clip_stats()
    assert got == want
    assert layer.clip_stats() == (0, 0)              # reading clears
    # the oracle takes the same decisions except for values within a BF16
    # step of the limit, which its exact h1 may round to the other side
    o = run_oracle(case, swiglu_limit=LIMIT, backward=False)
    oc = o["state"]["clip"]
    near = np.abs(np.abs(o["state"]["h1"]) - LIMIT) <= 2.0 ** -7
    slack = (int(near[:, :F].sum()), int(near[:, F:].sum()))
    assert abs(got[0] - oc[0]) <= slack[0] and abs(got[1] - oc[1]) <= slack[1]
    # two forwards accumulate
    x = case.x.to("cuda")
    ids = torch.from_numpy(case.ids).to("cuda")
    sc = torch.from_numpy(case.scores).to("cuda")
    for _ in range(2):
        layer.forward(x, ids, sc, g["W13"], g["W2"], saved=saved)
    assert layer.clip_stats() == (2 * want[0], 2 * want[1])
    # no limit: nothing counted
    g0 = run_gpu(case, backward=False)
    assert g0["layer"].clip_stats() == (0, 0)


def test_weights_1x32_prep_and_forward():
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    w = synth.Workload("w1x32", 160, 256, 384, 6, 2, "mxfp8", "uniform", seed=44)
    case = Case(w)
    dev = torch.device("cuda")
    pw = PreparedWeight(case.w2.to(dev), "mxfp8_1x32", with_transpose=False)
    E, N, K = pw.shape
    codes = pw.data.cpu().numpy()
    sf = unpack_weight_sf(pw.scale.cpu().numpy(), E * N, K).reshape(E, N, K // 32)
    q, e = fm.mx_quantize(to_f64(case.w2), axis=-1)
    np.testing.assert_array_equal(fm.e4m3_decode(codes), q)
    np.testing.assert_array_equal(sf.astype(np.int64) - 127, e)
    # forward with 1x32 weights vs the oracle with 1x32 blocks
    g = run_gpu(case, training=False, weight_prec="mxfp8_1x32")
    o = run_oracle(case, weight_blocks="1x32", backward=False)
    assert g["err_bits"] == 0
    assert rel_err(g["out"], o["out"]) <= TOL["mxfp8"]
    # ... and it is the 1x32 weight that was used: closer to the 1x32 oracle
    o32 = run_oracle(case, backward=False)
    assert rel_err(g["out"], o["out"]) < rel_err(g["out"], o32["out"])
    # the backward needs 32x32 weights with their transposed copy
    layer_t = MoELayer(case.T, w.D, w.F, w.E, w.K, "mxfp8", training=True)
    W13 = PreparedWeight(case.w13.to(dev), "mxfp8_1x32", with_transpose=False)
    saved = layer_t.new_saved()
    x = case.x.to(dev)
    ids = torch.from_numpy(case.ids).to(dev)
    sc = torch.from_numpy(case.scores).to(dev)
    layer_t.forward(x, ids, sc, W13, pw, saved=saved)
    with pytest.raises(abi.MoEError) as ei:
        layer_t.backward(saved, case.dy.to(dev), W13, pw)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    layer_t.close()
