"""moe_forward_static_scratch: the inference forward for callers that cannot
allocate device memory (it keeps its intermediates in the library's static
device array instead of a context's scratch).  Its output must match the
context-based moe_forward on the same inputs, on two calls in a row that
share the array.  This file is collected last on purpose."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth

from moe_cases import TOL, rel_err, to_f64

pytestmark = pytest.mark.gpu


def _inputs(w, T, dev):
    ids, scores = synth.make_routing(w)
    x = synth.make_tokens(w, dev)[:T].contiguous()
    return x, torch.from_numpy(ids[:T].copy()).to(dev), torch.from_numpy(scores[:T].copy()).to(dev)


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_static_scratch_forward_matches_context_forward(precision):
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    dev = torch.device("cuda")
    w = synth.Workload("noalloc", 160, 256, 256, 8, 2, precision, "topk_logits", inactive_frac=0.05, seed=41)
    w13, w2 = synth.make_weights(w, dev)
    W13 = PreparedWeight(w13, precision, with_transpose=False)
    W2 = PreparedWeight(w2, precision, with_transpose=False)
    layer = MoELayer(w.T, w.D, w.F, w.E, w.K, precision)
    cfg = abi.make_config(w.T, w.D, w.F, w.E, w.K, abi.MOE_MXFP8 if precision == "mxfp8" else abi.MOE_BF16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # two calls in a row with different inputs share (and overwrite) the static array
    for T, seed in ((160, 41), (97, 42)):
        ws = synth.scaled(w, seed=seed)
        x, ids, sc = _inputs(ws, T, dev)
        ref = layer.forward(x, ids, sc, W13, W2)
        got = torch.full_like(ref, float("nan"))
        abi.moe_forward_static_scratch(cfg, T, x, ids, sc, W13.struct, W2.struct, got, 0, err)
        torch.cuda.synchronize()
        assert rel_err(to_f64(got), to_f64(ref)) <= TOL[precision]
        assert not torch.isnan(got.float()).any()
    assert int(err.item()) == 0
    assert layer.error_bits() == 0
    layer.close()


def test_static_scratch_rejects_oversized_calls():
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import PreparedWeight
    dev = torch.device("cuda")
    w = synth.Workload("big", 8192, 1024, 256, 8, 8, "bf16", "uniform", seed=43)
    w13, w2 = synth.make_weights(w, dev)
    W13 = PreparedWeight(w13, "bf16", with_transpose=False)
    W2 = PreparedWeight(w2, "bf16", with_transpose=False)
    cfg = abi.make_config(w.T, w.D, w.F, w.E, w.K, abi.MOE_BF16)
    x = torch.zeros((w.T, w.D), dtype=torch.bfloat16, device=dev)
    ids = torch.zeros((w.T, w.K), dtype=torch.int32, device=dev)
    sc = torch.zeros((w.T, w.K), dtype=torch.float32, device=dev)
    out = torch.zeros((w.T, w.D), dtype=torch.bfloat16, device=dev)
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_forward_static_scratch(cfg, w.T, x, ids, sc, W13.struct, W2.struct, out)
    assert ei.value.status == abi.MOE_ERR_CAPACITY
    assert torch.count_nonzero(out).item() == 0
