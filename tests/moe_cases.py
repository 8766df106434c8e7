"""Shared helpers of the parity tests: seeded cases, the CUDA path through the
C ABI, and the oracle on the same inputs.

Inputs come from the seeded generator only; expected values come from the
oracle only.
"""

import numpy as np
import torch

from mixture_experts_routed_route_gb300 import synth

TOL = {"bf16": 1e-2, "mxfp8": 3e-2}   # max|gpu - ref| / max|ref|


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / den)


def to_f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def bf16_from_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


class Case:
    """One seeded workload: inputs on the CPU (torch) and their fp64 copies."""

    def __init__(self, w, T=None, ids=None, scores=None, seed_layer=0):
        self.w = w
        self.T = w.T if T is None else T
        if ids is None:
            ids, scores = synth.make_routing(w, layer=seed_layer)
        self.ids = np.ascontiguousarray(ids[: self.T]).astype(np.int32)
        self.scores = np.ascontiguousarray(scores[: self.T]).astype(np.float32)
        self.x = synth.make_tokens(w, "cpu", layer=seed_layer)[: self.T].contiguous()
        self.dy = synth.make_grad_out(w, "cpu", layer=seed_layer)[: self.T].contiguous()
        self.w13, self.w2 = synth.make_weights(w, "cpu", layer=seed_layer)

    # fp64 views for the oracle
    def oracle_inputs(self):
        return (to_f64(self.x), self.ids.astype(np.int64), self.scores, to_f64(self.w13), to_f64(self.w2))


def run_gpu(case, precision=None, training=True, debug=False, out_init=None, max_tokens=None,
            dx_init=None, dw_fp32=False, backward=True):
    """Forward (and backward) of a case through the C ABI; returns a dict of
    host arrays plus the layer object for further inspection."""
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight

    w = case.w
    precision = precision or w.precision
    dev = torch.device("cuda")
    T = case.T
    layer = MoELayer(max_tokens or max(T, 1), w.D, w.F, w.E, w.K, precision, training=training, debug=debug)
    W13 = PreparedWeight(case.w13.to(dev), precision, with_transpose=training)
    W2 = PreparedWeight(case.w2.to(dev), precision, with_transpose=training)
    x = case.x.to(dev)
    ids = torch.from_numpy(case.ids).to(dev)
    sc = torch.from_numpy(case.scores).to(dev)
    out = torch.zeros((T, w.D), dtype=torch.bfloat16, device=dev)
    acc = out_init is not None
    if acc:
        out.copy_(out_init)
    saved = layer.new_saved() if training else None
    layer.forward(x, ids, sc, W13, W2, out=out, saved=saved, accumulate=acc)
    res = {"layer": layer, "W13": W13, "W2": W2, "saved": saved, "out": to_f64(out), "out_t": out}
    if training and backward:
        dy = case.dy.to(dev)
        dx = torch.zeros((T, w.D), dtype=torch.bfloat16, device=dev)
        if dx_init is not None:
            dx.copy_(dx_init)
        dx, dW13, dW2 = layer.backward(saved, dy, W13, W2, dx=dx, accumulate_dx=dx_init is not None,
                                       dw_fp32=dw_fp32)
        res.update(dx=to_f64(dx), dW13=to_f64(dW13), dW2=to_f64(dW2))
    torch.cuda.synchronize()
    res["err_bits"] = layer.error_bits()
    return res


def run_oracle(case, precision=None, out_init=None, dx_init=None, dw_fp32=False, backward=True):
    from oracle import moe
    precision = precision or case.w.precision
    x, ids, s, w13, w2 = case.oracle_inputs()
    st = moe.forward(x, ids, s, w13, w2, precision, out_init=out_init)
    res = {"state": st, "out": st["out"]}
    if backward:
        g = moe.backward(st, to_f64(case.dy), w13, w2, dx_init=dx_init, dw_fp32=dw_fp32)
        res.update(dx=g["dX"], dW13=g["dW13"], dW2=g["dW2"], grads=g)
    return res
