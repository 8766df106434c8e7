"""Full-size parity at the 384-expert, D=7168 shape, in the launch sequence
the benchmark times (BF16 shared expert first, then the MXFP8 routed layer
accumulating onto it, forward and backward).

The oracle cannot run the whole layer in fp64 in seconds, so it checks
sampled outputs it can compute one by one: a few tokens are drawn, the
experts their active routes reach form an oracle sample (routes to other
experts disabled; each kept expert keeps exactly its rows), and the GPU's
out and dX of those tokens and dW13/dW2 of those experts are compared.  The
routing arrays are compared in full, bit-exact."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth
from oracle import moe as omoe
from oracle import sample as osample

from moe_cases import TOL, check_mx_wgrad, rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def full_run():
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    w = synth.WORKLOADS["e384_mxfp8_zipf_train"]
    dev = torch.device("cuda")
    T, D, F, E, K = w.T, w.D, w.F, w.E, w.K
    ids, scores = synth.make_routing(w)
    x = synth.make_tokens(w, dev)
    dy = synth.make_grad_out(w, dev)
    w13, w2 = synth.make_weights(w, dev)
    sw13, sw2 = synth.make_shared_weights(w, dev)
    W13, W2 = PreparedWeight(w13, "mxfp8"), PreparedWeight(w2, "mxfp8")
    sW13, sW2 = PreparedWeight(sw13, "bf16"), PreparedWeight(sw2, "bf16")
    layer = MoELayer(T, D, F, E, K, "mxfp8", training=True)
    shared = MoELayer(T, D, w.shared_F, 1, 1, "bf16", training=True)
    saved, s_saved = layer.new_saved(), shared.new_saved()
    s_ids = torch.zeros((T, 1), dtype=torch.int32, device=dev)
    s_sc = torch.ones((T, 1), dtype=torch.float32, device=dev)
    ids_d, sc_d = torch.from_numpy(ids).to(dev), torch.from_numpy(scores).to(dev)
    out = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    shared.forward(x, s_ids, s_sc, sW13, sW2, out=out, saved=s_saved)
    layer.forward(x, ids_d, sc_d, W13, W2, out=out, saved=saved, accumulate=True)
    shared.backward(s_saved, dy, sW13, sW2, dx=dx)
    _, dW13, dW2 = layer.backward(saved, dy, W13, W2, dx=dx, accumulate_dx=True)
    torch.cuda.synchronize()
    assert layer.error_bits() == 0 and shared.error_bits() == 0

    rng = np.random.default_rng(2024)
    tokens = sorted(rng.choice(T, size=3, replace=False).tolist())
    experts = sorted(set(int(e) for t in tokens for e in ids[t] if e >= 0))
    hdr = layer.saved_field(saved, abi.MOE_SAVED_HEADER, torch.int32, (16,)).cpu().numpy()
    fields = {f: layer.saved_field(saved, f, torch.int32, (n,)).cpu().numpy()
              for f, n in ((abi.MOE_SAVED_COUNTS, E), (abi.MOE_SAVED_POFFSETS, E + 1),
                           (abi.MOE_SAVED_PERM, int(hdr[2])), (abi.MOE_SAVED_INV, T * K))}
    res = dict(w=w, ids=ids, scores=scores, tokens=tokens, experts=experts, hdr=hdr, fields=fields,
               out=to_f64(out[tokens]), dx=to_f64(dx[tokens]),
               dW13=to_f64(dW13[experts]), dW2=to_f64(dW2[experts]),
               x=to_f64(x), dy=to_f64(dy), w13=to_f64(w13[experts]), w2=to_f64(w2[experts]),
               sw13=to_f64(sw13), sw2=to_f64(sw2))
    return res


def test_fullsize_routing_bit_exact(full_run):
    from mixture_experts_routed_route_gb300 import abi
    r = full_run
    rt = omoe.route(r["ids"], r["w"].E)
    assert r["hdr"][2] == rt.poffsets[-1] and r["hdr"][3] == rt.num_active
    np.testing.assert_array_equal(r["fields"][abi.MOE_SAVED_COUNTS], rt.counts)
    np.testing.assert_array_equal(r["fields"][abi.MOE_SAVED_POFFSETS], rt.poffsets)
    np.testing.assert_array_equal(r["fields"][abi.MOE_SAVED_PERM], rt.perm)
    np.testing.assert_array_equal(r["fields"][abi.MOE_SAVED_INV], rt.inv)


def test_fullsize_sampled_outputs_and_gradients(full_run):
    r = full_run
    tok = r["tokens"]
    # shared expert (BF16, dense) on the sampled tokens only: every quantity is row-local
    one = np.zeros((len(tok), 1), np.int64)
    ones = np.ones((len(tok), 1), np.float32)
    sst = omoe.forward(r["x"][tok], one, ones, r["sw13"], r["sw2"], "bf16")
    sgr = omoe.backward(sst, r["dy"][tok], r["sw13"], r["sw2"])
    init_out = np.zeros_like(r["x"])
    init_out[tok] = sst["out"]
    init_dx = np.zeros_like(r["x"])
    init_dx[tok] = sgr["dX"]
    sub_ids = osample.restrict_routes(r["ids"], r["experts"])
    st = omoe.forward(r["x"], sub_ids, r["scores"], r["w13"], r["w2"], "mxfp8", out_init=init_out)
    gr = omoe.backward(st, r["dy"], r["w13"], r["w2"], dx_init=init_dx)
    assert rel_err(r["out"], st["out"][tok]) <= TOL["mxfp8"]
    assert rel_err(r["dx"], gr["dX"][tok]) <= TOL["mxfp8"]
    # weight gradients: the stated tolerance on every code both sides decide
    # alike, plus exactly the contribution of codes that lie on a rounding
    # decision within the FP32 spread (see moe_cases.check_mx_wgrad)
    errs = check_mx_wgrad(r["dW13"], r["dW2"], st, gr)
    assert np.median([e for pair in errs for e in pair]) <= TOL["mxfp8"] / 3
