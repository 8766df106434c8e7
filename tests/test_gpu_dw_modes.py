"""The weight-gradient output modes against each other, bit for bit, on the
same saved state ("Dist-MoE: Speed-of-light distributed Mixture-of-Experts
kernels", section 05: the weight gradients are stored in BF16 or FP32):

* BF16 overwrite (the tensor-store epilogue) is the reference;
* FP32 overwrite, rounded to BF16 to nearest-even, equals it;
* FP32 accumulate equals init + the FP32 gradient (one FP32 add);
* BF16 accumulate equals bf16(init + the FP32 gradient);
* an expert no route reaches gets zeros, or keeps its old values when
  accumulating.

All four go through the same GEMM and differ in the epilogue: BF16 and FP32
overwrite stage the tile in shared memory and store it with TMA, FP32
accumulate stages it and adds it with a TMA reduce-add (the one FP32 add is
formed in L2), BF16 accumulate uses plain stores (it rounds old + new once)."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth

from moe_cases import Case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_dw_modes_agree(precision):
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    # 24 experts with Zipf routing over 96 tokens: 5 experts get no route
    w = synth.Workload(f"dw_modes_{precision}", 96, 256, 384, 24, 2, precision, "zipf", inactive_frac=0.1,
                       zipf_s=1.4, seed=31)
    case = Case(w)
    dev = torch.device("cuda")
    layer = MoELayer(case.T, w.D, w.F, w.E, w.K, precision, training=True)
    W13 = PreparedWeight(case.w13.to(dev), precision, with_transpose=True)
    W2 = PreparedWeight(case.w2.to(dev), precision, with_transpose=True)
    saved = layer.new_saved()
    layer.forward(case.x.to(dev), torch.from_numpy(case.ids).to(dev), torch.from_numpy(case.scores).to(dev),
                  W13, W2, saved=saved)
    dy = case.dy.to(dev)

    def bwd(dt, acc, init=None):
        dW13 = torch.empty((w.E, 2 * w.F, w.D), dtype=dt, device=dev)
        dW2 = torch.empty((w.E, w.D, w.F), dtype=dt, device=dev)
        if init is not None:
            dW13.copy_(init[0])
            dW2.copy_(init[1])
        _, a, b = layer.backward(saved, dy, W13, W2, dW13=dW13, dW2=dW2, dw_fp32=dt == torch.float32,
                                 dw_accumulate=acc)
        return a, b

    ref13, ref2 = bwd(torch.bfloat16, False)
    f13, f2 = bwd(torch.float32, False)
    rng = np.random.default_rng(32)
    i13 = torch.from_numpy(rng.normal(size=(w.E, 2 * w.F, w.D))).to(torch.float32).to(dev)
    i2 = torch.from_numpy(rng.normal(size=(w.E, w.D, w.F))).to(torch.float32).to(dev)
    a13, a2 = bwd(torch.float32, True, (i13, i2))
    b13, b2 = bwd(torch.bfloat16, True, (i13.to(torch.bfloat16), i2.to(torch.bfloat16)))
    torch.cuda.synchronize()
    assert layer.error_bits() == 0

    assert torch.equal(f13.to(torch.bfloat16), ref13) and torch.equal(f2.to(torch.bfloat16), ref2)
    assert torch.equal(a13, i13 + f13) and torch.equal(a2, i2 + f2)
    want13 = (i13.to(torch.bfloat16).float() + f13).to(torch.bfloat16)
    want2 = (i2.to(torch.bfloat16).float() + f2).to(torch.bfloat16)
    assert torch.equal(b13, want13) and torch.equal(b2, want2)

    hit = np.zeros(w.E, bool)
    hit[case.ids[case.ids >= 0]] = True
    assert (~hit).any(), "the case should leave some expert without routes"
    idle = torch.from_numpy(~hit).to(dev)
    assert torch.all(ref13[idle] == 0) and torch.all(f2[idle] == 0)
    assert torch.equal(a13[idle], i13[idle]) and torch.equal(b2[idle], i2[idle].to(torch.bfloat16))
    assert torch.any(ref13[~idle] != 0)
    layer.close()
