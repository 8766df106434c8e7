"""Save-or-replay of the expert state ("Dist-MoE: Speed-of-light distributed
Mixture-of-Experts kernels", section 04 "Activation Packing and Dynamic
Recompute": a layer that cannot keep its full state keeps its input, and
the backward rebuilds the rest):

* a backward that replays an input-only forward gives the same gradients,
  bit for bit, as one that reads the full saved state (the replay runs the
  forward's own kernels on the same inputs), BF16 and MXFP8, with the score
  gradient; and they agree with the fp64 oracle;
* a stack of three layers in one ActivationSlot whose capacity makes the
  planner keep the first layer's full state and replay the other two; each
  layer's gradients equal its full-state gradients;
* the same stack captured as one CUDA graph and replayed with new inputs;
* the post-expert RMSNorm on an input-only state;
* argument errors (host-side, nothing launched): replay flags on a context
  without MOE_REPLAY, a backward flag that does not match the forward.
"""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import abi, synth
from oracle import slot_plan as sp

from moe_cases import TOL, Case, rel_err, run_oracle, to_f64

pytestmark = pytest.mark.gpu

D, F, E, K = 256, 256, 8, 2


def _workload(precision, seed, T=192):
    return synth.Workload(f"replay_{precision}", T, D, F, E, K, precision, "zipf", inactive_frac=0.05,
                          zipf_s=1.2, seed=seed)


def _weights(case, precision):
    from mixture_experts_routed_route_gb300.layer import PreparedWeight
    dev = torch.device("cuda")
    return (PreparedWeight(case.w13.to(dev), precision, with_transpose=True),
            PreparedWeight(case.w2.to(dev), precision, with_transpose=True))


class _Io:
    """Device inputs and outputs of one layer (fixed addresses)."""

    def __init__(self, T):
        dev = torch.device("cuda")
        self.x = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
        self.ids = torch.empty((T, K), dtype=torch.int32, device=dev)
        self.sc = torch.empty((T, K), dtype=torch.float32, device=dev)
        self.dy = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
        self.dW13 = torch.empty((E, 2 * F, D), dtype=torch.bfloat16, device=dev)
        self.dW2 = torch.empty((E, D, F), dtype=torch.bfloat16, device=dev)
        self.dp = torch.empty((T, K), dtype=torch.float32, device=dev)

    def load(self, case):
        self.x.copy_(case.x)
        self.ids.copy_(torch.from_numpy(case.ids))
        self.sc.copy_(torch.from_numpy(case.scores))
        self.dy.copy_(case.dy)
        self.dp.fill_(float("nan"))   # every entry must be written

    def forward(self, layer, W, saved, input_only):
        layer.forward(self.x, self.ids, self.sc, *W, out=self.out, saved=saved, save_input_only=input_only)

    def backward(self, layer, W, saved, input_only):
        layer.backward(saved, self.dy, *W, dx=self.dx, dW13=self.dW13, dW2=self.dW2, d_scores=self.dp,
                       replay=input_only)

    def results(self):
        return {k: getattr(self, k).clone() for k in ("out", "dx", "dW13", "dW2", "dp")}


def _assert_same(a, b):
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_replay_equals_full_state(precision):
    from mixture_experts_routed_route_gb300.layer import MoELayer
    case = Case(_workload(precision, 71))
    layer = MoELayer(case.T, D, F, E, K, precision, training=True, replay=True)
    W = _weights(case, precision)
    io = _Io(case.T)
    io.load(case)
    full_saved = layer.new_saved()
    io.forward(layer, W, full_saved, False)
    io.backward(layer, W, full_saved, False)
    full = io.results()
    io.load(case)
    sv = layer.new_saved(input_only=True)
    assert sv.numel() < full_saved.numel() / 4
    io.forward(layer, W, sv, True)
    io.backward(layer, W, sv, True)
    rep = io.results()
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    _assert_same(full, rep)
    # the input-only state holds the routing and a copy of x
    xs = layer.saved_field(sv, abi.MOE_SAVED_X, torch.bfloat16, (case.T, D), input_only=True)
    assert torch.equal(xs.cpu(), case.x)
    perm_full = layer.saved_field(full_saved, abi.MOE_SAVED_PERM, torch.int32, (layer.r_cap,))
    perm_in = layer.saved_field(sv, abi.MOE_SAVED_PERM, torch.int32, (layer.r_cap,), input_only=True)
    n_rows = int(layer.saved_field(sv, abi.MOE_SAVED_HEADER, torch.int32, (16,), input_only=True)[2])
    assert torch.equal(perm_full[:n_rows], perm_in[:n_rows])
    # and the replayed gradients against the fp64 oracle
    o = run_oracle(case)
    for k in ("out", "dx", "dp") if precision == "mxfp8" else ("out", "dx", "dp", "dW13", "dW2"):
        assert rel_err(to_f64(rep[k]), o[k]) <= TOL[precision], k
    layer.close()


def test_slot_stack_replays_and_matches_full_state():
    from mixture_experts_routed_route_gb300.layer import ActivationSlot, MoELayer
    precision = "mxfp8"
    w = _workload(precision, 81)
    cases = [Case(w, seed_layer=l) for l in range(3)]
    layer = MoELayer(w.T, D, F, E, K, precision, training=True, replay=True)
    Ws = [_weights(c, precision) for c in cases]
    full_b = abi.moe_saved_state_bytes(layer.cfg)
    in_b = abi.moe_saved_input_bytes(layer.cfg)
    cap = sp.align128(full_b) + 2 * sp.align128(in_b)     # room for one full state and two inputs
    want = sp.plan_stack([(full_b, in_b)] * 3, cap)
    assert [p["decision"] for p in want] == [sp.FULL, sp.INPUT, sp.INPUT]

    # each layer alone, full state
    io = _Io(w.T)
    ref = []
    for c, W in zip(cases, Ws):
        io.load(c)
        s = layer.new_saved()
        io.forward(layer, W, s, False)
        io.backward(layer, W, s, False)
        ref.append(io.results())

    # the stack: forwards in order, backwards in reverse, states in one slot
    slot = ActivationSlot(cap, max_layers=4)
    ios = [_Io(w.T) for _ in cases]
    states = []
    for l, (c, W) in enumerate(zip(cases, Ws)):
        ios[l].load(c)
        saved, input_only = slot.push(layer, 2 - l)
        assert input_only == (want[l]["decision"] == sp.INPUT)
        ios[l].forward(layer, W, saved, input_only)
        states.append((saved, input_only))
    for l in reversed(range(3)):
        saved, input_only = states[l]
        ios[l].backward(layer, Ws[l], saved, input_only)
        slot.pop(saved)
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    assert slot.slot.layers == 0 and slot.slot.cursor == 0
    for l in range(3):
        _assert_same(ref[l], ios[l].results())
    layer.close()


def test_slot_stack_in_a_cuda_graph():
    """Decisions and offsets do not depend on the routing, so one captured
    graph of the stack replays with new inputs."""
    from mixture_experts_routed_route_gb300.layer import ActivationSlot, MoELayer
    precision = "bf16"
    w = _workload(precision, 91, T=128)
    layer = MoELayer(w.T, D, F, E, K, precision, training=True, replay=True)
    W = _weights(Case(w), precision)
    full_b = abi.moe_saved_state_bytes(layer.cfg)
    in_b = abi.moe_saved_input_bytes(layer.cfg)
    slot = ActivationSlot(sp.align128(full_b) + sp.align128(in_b), max_layers=2)
    ios = [_Io(w.T) for _ in range(2)]
    states = [slot.push(layer, 1), slot.push(layer, 0)]
    assert [s[1] for s in states] == [False, True]

    def step():
        for l in range(2):
            ios[l].forward(layer, W, states[l][0], states[l][1])
        for l in reversed(range(2)):
            ios[l].backward(layer, W, states[l][0], states[l][1])

    first = [Case(w, seed_layer=l) for l in range(2)]
    for l in range(2):
        ios[l].load(first[l])
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for r in (1, 2):
        cases = [Case(w, seed_layer=10 * r + l) for l in range(2)]
        for l in range(2):
            ios[l].load(cases[l])
        graph.replay()
        torch.cuda.synchronize()
        assert layer.error_bits() == 0
        got = [io.results() for io in ios]
        # eager, full state, same inputs
        for l in range(2):
            ios[l].load(cases[l])
            s = layer.new_saved()
            ios[l].forward(layer, W, s, False)
            ios[l].backward(layer, W, s, False)
            _assert_same(ios[l].results(), got[l])
    del graph
    layer.close()


def test_post_norm_with_an_input_only_state():
    from mixture_experts_routed_route_gb300.layer import MoELayer
    precision = "mxfp8"
    case = Case(_workload(precision, 95))
    gamma = torch.from_numpy(np.random.default_rng(96).normal(1.0, 0.25, size=D)).to(torch.bfloat16).cuda()
    layer = MoELayer(case.T, D, F, E, K, precision, training=True, post_norm=True, replay=True)
    layer.set_post_norm(gamma, 1e-5)
    W = _weights(case, precision)
    io = _Io(case.T)
    res = []
    for input_only in (False, True):
        io.load(case)
        s = layer.new_saved(input_only=input_only)
        io.forward(layer, W, s, input_only)
        dxp, dg = layer.post_norm_backward(s, io.dy)
        io.dy.copy_(dxp)
        io.backward(layer, W, s, input_only)
        r = io.results()
        r["dgamma"] = dg.clone()
        r["prenorm"] = layer.saved_field(s, abi.MOE_SAVED_PRENORM, torch.bfloat16, (case.T, D),
                                         input_only=input_only).clone()
        res.append(r)
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    _assert_same(res[0], res[1])
    layer.close()


def test_replay_argument_errors():
    from mixture_experts_routed_route_gb300.layer import MoELayer
    precision = "bf16"
    case = Case(_workload(precision, 99, T=64))
    W = _weights(case, precision)
    io = _Io(case.T)
    io.load(case)
    plain = MoELayer(case.T, D, F, E, K, precision, training=True)      # no MOE_REPLAY
    with pytest.raises(abi.MoEError) as ei:
        io.forward(plain, W, plain.new_saved(input_only=True), True)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    s = plain.new_saved()
    io.forward(plain, W, s, False)
    with pytest.raises(abi.MoEError) as ei:
        io.backward(plain, W, s, True)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG

    layer = MoELayer(case.T, D, F, E, K, precision, training=True, replay=True)
    with pytest.raises(abi.MoEError):                 # inference forward cannot save an input
        layer.forward(io.x, io.ids, io.sc, *W, out=io.out, saved=None, save_input_only=True)
    full = layer.new_saved()
    io.forward(layer, W, full, False)
    with pytest.raises(abi.MoEError) as ei:           # replay flag on a full state
        io.backward(layer, W, full, True)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    inp = layer.new_saved(input_only=True)
    io.forward(layer, W, inp, True)
    with pytest.raises(abi.MoEError) as ei:           # no replay flag on an input-only state
        io.backward(layer, W, inp, False)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    io.backward(layer, W, inp, True)                  # the matching call still works
    torch.cuda.synchronize()
    assert layer.error_bits() == 0 and plain.error_bits() == 0
    plain.close()
    layer.close()
