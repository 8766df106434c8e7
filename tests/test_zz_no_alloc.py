"""moe_forward_static_scratch: the inference forward for callers that cannot
allocate device memory when they need the layer (an engine that gave all
free HBM to its KV cache, a plugin handed a stream but no allocator, a loop
that must not call cudaMalloc because it can synchronise the device).  It
keeps its intermediates in the library's static device array instead of a
context's scratch, and launches the same kernels in the same configuration
as an inference moe_forward, so its output must equal moe_forward's bit for
bit, on two calls in a row that share (and overwrite) the array.  This file
is collected last on purpose."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth

pytestmark = pytest.mark.gpu


def _inputs(w, T, dev):
    ids, scores = synth.make_routing(w)
    x = synth.make_tokens(w, dev)[:T].contiguous()
    return x, torch.from_numpy(ids[:T].copy()).to(dev), torch.from_numpy(scores[:T].copy()).to(dev)


def _prec_code(precision):
    from mixture_experts_routed_route_gb300 import abi
    return abi.MOE_MXFP8 if precision.startswith("mxfp8") else abi.MOE_BF16


def _run_pair(w, precision, weight_prec, calls, accumulate=False):
    """For each (T, seed): moe_forward through a context and the static
    forward on the same inputs; asserts bitwise equality."""
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    dev = torch.device("cuda")
    w13, w2 = synth.make_weights(w, dev)
    W13 = PreparedWeight(w13, weight_prec, with_transpose=False)
    W2 = PreparedWeight(w2, weight_prec, with_transpose=False)
    del w13, w2
    tmax = max(T for T, _ in calls)
    layer = MoELayer(tmax, w.D, w.F, w.E, w.K, precision)
    cfg = abi.make_config(tmax, w.D, w.F, w.E, w.K, _prec_code(precision))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flags = abi.MOE_ACCUMULATE_OUT if accumulate else 0
    for T, seed in calls:
        x, ids, sc = _inputs(synth.scaled(w, seed=seed), T, dev)
        base = (torch.randn((T, w.D), generator=torch.Generator(device=dev).manual_seed(seed), device=dev)
                .to(torch.bfloat16) if accumulate else torch.zeros((T, w.D), dtype=torch.bfloat16, device=dev))
        ref = base.clone()
        layer.forward(x, ids, sc, W13, W2, out=ref, accumulate=accumulate)
        got = base.clone() if accumulate else torch.full_like(ref, float("nan"))
        abi.moe_forward_static_scratch(cfg, T, x, ids, sc, W13.struct, W2.struct, got, err, flags)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (T, seed)
        assert torch.count_nonzero(ref.float()).item() > 0
    assert int(err.item()) == 0
    assert layer.error_bits() == 0
    layer.close()


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_static_scratch_forward_equals_context_forward(precision):
    w = synth.Workload("noalloc", 160, 256, 256, 8, 2, precision, "topk_logits", inactive_frac=0.05, seed=41)
    _run_pair(w, precision, precision, ((160, 41), (97, 42)))


def test_static_scratch_with_1x32_weights_and_accumulate():
    w = synth.Workload("noalloc_1x32", 128, 512, 256, 6, 3, "mxfp8", "zipf", inactive_frac=0.1, seed=44)
    _run_pair(w, "mxfp8", "mxfp8_1x32", ((128, 44), (33, 45)), accumulate=True)


def test_static_scratch_decode_at_the_e384_shape():
    """One and eight tokens at D=7168, F=2048, E=384, K=6 in MXFP8: the
    array holds the rows of the experts a step can reach, not 31 pad rows
    for every expert."""
    w = synth.Workload("noalloc_decode", 8, 7168, 2048, 384, 6, "mxfp8", "uniform", seed=45)
    _run_pair(w, "mxfp8", "mxfp8", ((1, 45), (8, 46)))


def test_static_scratch_reports_device_errors_and_needs_an_error_word():
    """Bad expert IDs set the bad-ID bit in the caller's error word (the
    routes count as inactive, as in moe_forward); a call without an error
    word is refused before any launch."""
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import PreparedWeight
    dev = torch.device("cuda")
    w = synth.Workload("noalloc_err", 64, 256, 256, 4, 2, "bf16", "uniform", seed=47)
    w13, w2 = synth.make_weights(w, dev)
    W13 = PreparedWeight(w13, "bf16", with_transpose=False)
    W2 = PreparedWeight(w2, "bf16", with_transpose=False)
    cfg = abi.make_config(w.T, w.D, w.F, w.E, w.K, abi.MOE_BF16)
    x, ids, sc = _inputs(w, w.T, dev)
    ids[3, 1] = w.E + 5
    out = torch.zeros((w.T, w.D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    abi.moe_forward_static_scratch(cfg, w.T, x, ids, sc, W13.struct, W2.struct, out, err)
    torch.cuda.synchronize()
    assert int(err.item()) & abi.MOE_DEV_ERR_BAD_ID
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_forward_static_scratch(cfg, w.T, x, ids, sc, W13.struct, W2.struct, out, None)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG


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
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_forward_static_scratch(cfg, w.T, x, ids, sc, W13.struct, W2.struct, out, err)
    assert ei.value.status == abi.MOE_ERR_CAPACITY
    assert torch.count_nonzero(out).item() == 0
