"""Parity of the inference forward at the pages' own workload shapes, and of
the plain MXFP8 inference forward (32x32 weights, no saved state) on small
cases, against the oracle.

* ``e64_bf16``: T=2048, D=2048, F=1408, E=64, K=6, BF16, uniform routing.
  F/128 = 11 output tiles per expert and 64-row remainder blocks; the oracle
  runs the whole layer.
* ``e384_mxfp8``: T=2048, D=7168, F=2048, E=384, K=6, MXFP8 routed experts
  accumulated onto one dense BF16 shared expert (F=2048), uniform routing,
  inference (no saved state: the row-only gather and the context's routing
  copy).  The routing is compared in full, bit-exact; out on sampled tokens
  whose experts form an oracle sample.
* small MXFP8 and BF16 cases with ``training=False``.
"""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth
from oracle import moe as omoe
from oracle import sample as osample

from moe_cases import TOL, Case, assert_routing, ctx_routing, rel_err, run_gpu, run_oracle, to_f64

pytestmark = pytest.mark.gpu


def test_e64_bf16_inference_forward_matches_oracle():
    case = Case(synth.WORKLOADS["e64_bf16"])
    g = run_gpu(case, training=False, backward=False)
    assert g["err_bits"] == 0
    assert_routing(ctx_routing(g["layer"], case.T), case.ids.astype(np.int64), case.w.E)
    o = run_oracle(case, backward=False)
    assert rel_err(g["out"], o["out"]) <= TOL["bf16"]
    g["layer"].close()


@pytest.mark.parametrize("training", [False, True])
def test_e64_bf16_forward_tiles_and_remainders(training):
    """The same shape through the training forward too (row + column gather,
    saved h1), so both gathers meet F = 11 tiles of 128 and 64-row blocks."""
    case = Case(synth.WORKLOADS["e64_bf16"], T=512)
    g = run_gpu(case, training=training, backward=False)
    assert g["err_bits"] == 0
    o = run_oracle(case, backward=False)
    assert rel_err(g["out"], o["out"]) <= TOL["bf16"]
    g["layer"].close()


def test_e384_mxfp8_inference_shared_then_routed():
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    w = synth.WORKLOADS["e384_mxfp8"]
    dev = torch.device("cuda")
    T, D, F, E, K = w.T, w.D, w.F, w.E, w.K
    ids, scores = synth.make_routing(w)
    x = synth.make_tokens(w, dev)
    w13, w2 = synth.make_weights(w, dev)
    sw13, sw2 = synth.make_shared_weights(w, dev)
    W13 = PreparedWeight(w13, "mxfp8", with_transpose=False)
    W2 = PreparedWeight(w2, "mxfp8", with_transpose=False)
    sW13 = PreparedWeight(sw13, "bf16", with_transpose=False)
    sW2 = PreparedWeight(sw2, "bf16", with_transpose=False)
    layer = MoELayer(T, D, F, E, K, "mxfp8", training=False)
    shared = MoELayer(T, D, w.shared_F, 1, 1, "bf16", training=False)
    out = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    shared.forward(x, torch.zeros((T, 1), dtype=torch.int32, device=dev),
                   torch.ones((T, 1), dtype=torch.float32, device=dev), sW13, sW2, out=out)
    layer.forward(x, torch.from_numpy(ids).to(dev), torch.from_numpy(scores).to(dev), W13, W2, out=out,
                  accumulate=True)
    torch.cuda.synchronize()
    assert layer.error_bits() == 0 and shared.error_bits() == 0
    assert_routing(ctx_routing(layer, T), ids.astype(np.int64), E)

    rng = np.random.default_rng(77)
    tokens = sorted(rng.choice(T, size=4, replace=False).tolist())
    experts = sorted(set(int(e) for t in tokens for e in ids[t] if e >= 0))
    xf = to_f64(x)
    one = np.zeros((len(tokens), 1), np.int64)
    sst = omoe.forward(xf[tokens], one, np.ones((len(tokens), 1), np.float32), to_f64(sw13), to_f64(sw2), "bf16")
    init = np.zeros_like(xf)
    init[tokens] = sst["out"]
    st = omoe.forward(xf, osample.restrict_routes(ids, experts), scores, to_f64(w13[experts]),
                      to_f64(w2[experts]), "mxfp8", out_init=init)
    assert rel_err(to_f64(out[tokens]), st["out"][tokens]) <= TOL["mxfp8"]
    layer.close()
    shared.close()


def _mx_small(name, seed, **kw):
    base = dict(T=160, D=256, F=384, E=6, K=3, precision="mxfp8", routing="zipf", inactive_frac=0.1, zipf_s=1.3)
    base.update(kw)
    return synth.Workload(name, seed=seed, **base)


SMALL = {
    "mx_32x32": lambda: _mx_small("mx_inf_a", 31),
    "mx_32x32_wide": lambda: _mx_small("mx_inf_b", 32, D=512, F=256, E=10, K=2, routing="uniform"),
    "bf16_inf": lambda: _mx_small("bf16_inf", 33, precision="bf16"),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_inference_forward_matches_oracle(name):
    case = Case(SMALL[name]())
    p = case.w.precision
    g = run_gpu(case, training=False, backward=False)
    assert g["err_bits"] == 0
    assert_routing(ctx_routing(g["layer"], case.T), case.ids.astype(np.int64), case.w.E)
    o = run_oracle(case, backward=False)
    assert rel_err(g["out"], o["out"]) <= TOL[p]
    dead = np.all(case.ids < 0, axis=1)
    assert np.all(g["out"][dead] == 0.0)
    g["layer"].close()


@pytest.mark.parametrize("name", ["mx_32x32", "bf16_inf"])
def test_inference_equals_training_forward(name):
    """An inference forward and a training forward run the same arithmetic:
    out is bit-identical."""
    case = Case(SMALL[name]())
    a = run_gpu(case, training=False, backward=False)
    b = run_gpu(case, training=True, backward=False)
    np.testing.assert_array_equal(a["out"], b["out"])
    a["layer"].close()
    b["layer"].close()
