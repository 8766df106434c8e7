"""Ten stacked MXFP8 layers (T=4096, D=7168, F=2048, E=384, K=8, each layer
with its own Zipf(s in [0.8, 1.5]) routing and inputs): the forwards of all
ten, then the backwards in reverse order, captured once as one CUDA graph on
one context with fixed-capacity scratch, and replayed twice with new inputs
written in place between the replays (the Dist-MoE explainer's
changed-input / stable-address CUDA-graph check, section 07).

The ten layers share one expert weight set (tied weights): ten independent
MXFP8 weight sets with the transposed copies the input-gradient GEMMs read
would need about 338 GB.  The weight gradients of the ten layers therefore
accumulate in one FP32 buffer (the first backward overwrites it, the other
nine add), which is the gradient of the tied weights.

Checks after each replay: every layer's routing bit-exact against the
oracle; sampled tokens' out and dX of two layers against the oracle's
bounded sample; after the first replay, the FP32 dW of one sampled expert,
summed over the ten layers, against the oracle's per-layer gradients with
the undecided-code allowance of moe_cases.check_mx_wgrad."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth
from oracle import moe as omoe
from oracle import sample as osample

from moe_cases import TOL, rel_err, to_f64

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS["ten_layer_graph"]


def _layer_inputs(layer, replay):
    """Seeded inputs of one layer for one replay (replay 1 = changed inputs)."""
    w = synth.scaled(W, seed=W.seed + 100 * replay)
    s = synth.layer_zipf_s(w, layer)
    ids, scores = synth.make_routing(w, layer=layer, zipf_s=s)
    x = synth.make_tokens(w, "cpu", layer=layer)
    dy = synth.make_grad_out(w, "cpu", layer=layer)
    return ids, scores, x, dy


def test_ten_layer_graph_changed_inputs():
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    dev = torch.device("cuda")
    T, D, F, E, K, L = W.T, W.D, W.F, W.E, W.K, W.layers
    w13, w2 = synth.make_weights(W, dev)
    W13, W2 = PreparedWeight(w13, "mxfp8"), PreparedWeight(w2, "mxfp8")
    host13, host2 = w13, w2            # kept for the oracle's sampled experts
    layer = MoELayer(T, D, F, E, K, "mxfp8", training=True)
    saved = [layer.new_saved() for _ in range(L)]
    x = [torch.empty((T, D), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    dy = [torch.empty((T, D), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    ids = [torch.empty((T, K), dtype=torch.int32, device=dev) for _ in range(L)]
    sc = [torch.empty((T, K), dtype=torch.float32, device=dev) for _ in range(L)]
    out = [torch.empty((T, D), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    dx = [torch.empty((T, D), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    dW13 = torch.empty((E, 2 * F, D), dtype=torch.float32, device=dev)
    dW2 = torch.empty((E, D, F), dtype=torch.float32, device=dev)

    def load_replay(r):
        host = [_layer_inputs(l, r) for l in range(L)]
        for l, (i, s, xx, yy) in enumerate(host):
            ids[l].copy_(torch.from_numpy(i))
            sc[l].copy_(torch.from_numpy(s))
            x[l].copy_(xx)
            dy[l].copy_(yy)
        return host

    def step():
        for l in range(L):
            layer.forward(x[l], ids[l], sc[l], W13, W2, out=out[l], saved=saved[l])
        for n, l in enumerate(reversed(range(L))):
            layer.backward(saved[l], dy[l], W13, W2, dx=dx[l], dW13=dW13, dW2=dW2, dw_fp32=True,
                           dw_accumulate=n > 0)

    load_replay(0)
    step()                                     # eager once: kernel attributes, warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    rng = np.random.default_rng(77)
    for r in (0, 1):
        host = load_replay(r)
        graph.replay()
        torch.cuda.synchronize()
        assert layer.error_bits() == 0
        # every layer's routing, bit-exact
        for l in range(L):
            rt = omoe.route(host[l][0], E)
            perm = layer.saved_field(saved[l], abi.MOE_SAVED_PERM, torch.int32, (int(rt.poffsets[E]),)).cpu().numpy()
            inv = layer.saved_field(saved[l], abi.MOE_SAVED_INV, torch.int32, (T * K,)).cpu().numpy()
            np.testing.assert_array_equal(perm, rt.perm)
            np.testing.assert_array_equal(inv, rt.inv)
        # sampled tokens of two layers: out and dX
        for l in (0, L - 1) if r == 0 else (L // 2,):
            i_l, s_l, x_l, dy_l = host[l]
            t = int(rng.choice(np.nonzero(np.all(i_l >= 0, axis=1))[0]))
            experts = sorted(set(int(e) for e in i_l[t]))
            w13s, w2s = to_f64(host13[experts]), to_f64(host2[experts])
            res = osample.run(to_f64(x_l), i_l, s_l, w13s, w2s, experts, "mxfp8", dY=to_f64(dy_l))
            assert rel_err(to_f64(out[l][t:t + 1]), res["out"][t:t + 1]) <= TOL["mxfp8"]
            assert rel_err(to_f64(dx[l][t:t + 1]), res["grads"]["dX"][t:t + 1]) <= TOL["mxfp8"]
        if r == 0:
            # one expert's FP32 weight gradient, summed over the ten layers
            e = int(rng.choice(np.nonzero(np.bincount(host[0][0][host[0][0] >= 0], minlength=E))[0]))
            w13s, w2s = to_f64(host13[[e]]), to_f64(host2[[e]])
            ref13 = np.zeros((2 * F, D))
            ref2 = np.zeros((D, F))
            allow13 = np.zeros_like(ref13)
            allow2 = np.zeros_like(ref2)
            from moe_cases import mx_wgrad_allowance
            for l in range(L):
                i_l, s_l, x_l, dy_l = host[l]
                res = osample.run(to_f64(x_l), i_l, s_l, w13s, w2s, [e], "mxfp8", dY=to_f64(dy_l))
                g, st = res["grads"], res["state"]
                ref13 += g["dW13"][0]
                ref2 += g["dW2"][0]
                a13, a2, _, _ = mx_wgrad_allowance(st, g, 0)
                allow13 += a13
                allow2 += a2
            got13, got2 = to_f64(dW13[e]), to_f64(dW2[e])
            assert np.all(np.abs(got13 - ref13) <= TOL["mxfp8"] * np.max(np.abs(ref13)) + allow13)
            assert np.all(np.abs(got2 - ref2) <= TOL["mxfp8"] * np.max(np.abs(ref2)) + allow2)
    layer.close()
