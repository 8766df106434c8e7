"""MN-major input-gradient operands: MXFP8 weights prepared without the
transposed copy of their codes (only the input-gradient scale atoms), so the
two input-gradient GEMMs read the forward codes MN-major ("Dist-MoE:
Speed-of-light distributed Mixture-of-Experts kernels", section 02,
"Quantization Axes for Forward and Backward": static 32x32 weights let the
forward and the input-gradient GEMM share qdata with distinct scale
orientations).

Every gradient must equal the one computed with the transposed copy bit for
bit (same codes, same scales, same contraction order), on shapes whose W13
input-gradient GEMM takes two weight tiles per stage (D % 256 == 0) and one
(D = 384), and at the 7168-wide shape; dX also against the oracle."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth

from moe_cases import TOL, Case, rel_err, run_oracle, to_f64

pytestmark = pytest.mark.gpu


def _backward_both_ways(case):
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    w = case.w
    dev = torch.device("cuda")
    layer = MoELayer(case.T, w.D, w.F, w.E, w.K, "mxfp8", training=True)
    w13, w2 = case.w13.to(dev), case.w2.to(dev)
    k13, k2 = PreparedWeight(w13, "mxfp8"), PreparedWeight(w2, "mxfp8")
    m13, m2 = PreparedWeight(w13, "mxfp8", mn_major=True), PreparedWeight(w2, "mxfp8", mn_major=True)
    assert m13.data_t is None and m2.data_t is None and m13.scale_t is not None
    saved = layer.new_saved()
    x, dy = case.x.to(dev), case.dy.to(dev)
    out = layer.forward(x, torch.from_numpy(case.ids).to(dev), torch.from_numpy(case.scores).to(dev), m13, m2,
                        saved=saved)
    res = {}
    for name, A, B in (("k", k13, k2), ("mn", m13, m2)):
        dp = torch.zeros((case.T, w.K), dtype=torch.float32, device=dev)
        dx, dW13, dW2 = layer.backward(saved, dy, A, B, d_scores=dp)
        torch.cuda.synchronize()
        res[name] = [t.clone() for t in (dx, dW13, dW2, dp)]
    assert layer.error_bits() == 0
    layer.close()
    return out, res


CASES = {
    "pairs": lambda: synth.Workload("mn_pairs", 200, 256, 384, 8, 2, "mxfp8", "zipf", inactive_frac=0.1,
                                    zipf_s=1.2, seed=71),
    "single_tiles": lambda: synth.Workload("mn_single", 160, 384, 256, 6, 3, "mxfp8", "topk_logits",
                                           inactive_frac=0.05, seed=72),
}


@pytest.mark.parametrize("name", list(CASES))
def test_mn_major_gradients_equal_transposed_copy(name):
    case = Case(CASES[name]())
    _, res = _backward_both_ways(case)
    for a, b in zip(res["k"], res["mn"]):
        bits = torch.int32 if a.dtype == torch.float32 else torch.int16
        assert torch.equal(a.view(bits), b.view(bits))
    o = run_oracle(case)
    assert rel_err(to_f64(res["mn"][0]), o["dx"]) <= TOL["mxfp8"]


def test_mn_major_at_the_7168_wide_shape():
    """T=128, D=7168, F=2048, E=24, K=6: both input-gradient GEMMs at the
    E=384 layer's widths (56 K-stages for W2's, 32 for W13's)."""
    case = Case(synth.WORKLOADS["profile_e24"])
    _, res = _backward_both_ways(case)
    assert torch.equal(res["k"][0].view(torch.int16), res["mn"][0].view(torch.int16))
    assert torch.equal(res["k"][1].view(torch.int16), res["mn"][1].view(torch.int16))
    assert torch.equal(res["k"][3].view(torch.int32), res["mn"][3].view(torch.int32))
