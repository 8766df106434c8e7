"""The single-launch MXFP8 inference forward (MOE_FUSED_LAUNCH: routing,
gather, W13 + SwiGLU, W2 and combine in one persistent grid whose CTAs wait
on readiness counters, "Dist-MoE: Speed-of-light distributed
Mixture-of-Experts kernels", section 05, "Kernel Pipelines: Staged and
Mega").

Its output must equal the staged forward's bit for bit (same routing, same
row-bundle codes, same GEMM stages, same fixed-order combine), and the
oracle's within the MXFP8 tolerance; its routing arrays must equal the
oracle's.  Also: a capped grid (each CTA walks many records), graph replays
with new inputs, accumulate-out, bad IDs, the all-inactive step, and a wait
that runs out under a short limit, which must return the timeout bit
promptly and leave the context usable."""

import time

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth
from oracle import moe as omoe
from oracle import sample as osample

from moe_cases import TOL, assert_routing, ctx_routing, rel_err, to_f64

pytestmark = pytest.mark.gpu


class Rig:
    """One inference context with prepared MXFP8 weights of a workload."""

    def __init__(self, w, weight_prec="mxfp8", max_tokens=None):
        from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
        self.w = w
        self.dev = torch.device("cuda")
        w13, w2 = synth.make_weights(w, self.dev)
        self.W13 = PreparedWeight(w13, weight_prec, with_transpose=False)
        self.W2 = PreparedWeight(w2, weight_prec, with_transpose=False)
        self.w13_bf16, self.w2_bf16 = w13, w2
        self.layer = MoELayer(max_tokens or w.T, w.D, w.F, w.E, w.K, "mxfp8")

    def inputs(self, T, seed):
        ws = synth.scaled(self.w, seed=seed)
        ids, scores = synth.make_routing(ws)
        x = synth.make_tokens(ws, self.dev)[:T].contiguous()
        return x, torch.from_numpy(ids[:T].copy()).to(self.dev), torch.from_numpy(scores[:T].copy()).to(self.dev)

    def run(self, x, ids, sc, fused, out=None, accumulate=False):
        from mixture_experts_routed_route_gb300 import abi
        T = x.shape[0]
        if out is None:
            out = torch.full((T, self.w.D), float("nan"), dtype=torch.bfloat16, device=self.dev)
        flags = (abi.MOE_FUSED_LAUNCH if fused else 0) | (abi.MOE_ACCUMULATE_OUT if accumulate else 0)
        abi.moe_forward(self.layer.ctx, T, x, ids, sc, self.W13.struct, self.W2.struct, out, None, flags, None)
        return out

    def routing(self, T):
        return ctx_routing(self.layer, T)

    def close(self):
        self.layer.close()


def _bits(t):
    return t.view(torch.int16)


def _assert_same(a, b):
    assert torch.equal(_bits(a), _bits(b))


@pytest.fixture(scope="module")
def e384():
    w = synth.Workload("fused_e384", 16, 7168, 2048, 384, 6, "mxfp8", "uniform", seed=51)
    rig = Rig(w)
    yield rig
    rig.close()


@pytest.mark.parametrize("T", [1, 16])
def test_fused_equals_staged_and_oracle_at_e384(e384, T):
    rig = e384
    x, ids, sc = rig.inputs(T, 51 + T)
    staged = rig.run(x, ids, sc, fused=False)
    torch.cuda.synchronize()
    fused = rig.run(x, ids, sc, fused=True)
    torch.cuda.synchronize()
    assert rig.layer.error_bits() == 0
    _assert_same(fused, staged)
    ids_np, sc_np = ids.cpu().numpy(), sc.cpu().numpy()
    assert_routing(rig.routing(T), ids_np.astype(np.int64), rig.w.E)
    # oracle on sampled tokens: the experts they reach form an oracle sample
    tokens = list(range(T)) if T <= 2 else sorted(np.random.default_rng(T).choice(T, 3, replace=False).tolist())
    experts = sorted(set(int(e) for t in tokens for e in ids_np[t] if e >= 0))
    st = omoe.forward(to_f64(x), osample.restrict_routes(ids_np, experts), sc_np, to_f64(rig.w13_bf16[experts]),
                      to_f64(rig.w2_bf16[experts]), "mxfp8")
    assert rel_err(to_f64(fused[tokens]), st["out"][tokens]) <= TOL["mxfp8"]


def _small(seed, **kw):
    base = dict(T=160, D=256, F=384, E=6, K=3, precision="mxfp8", routing="zipf", inactive_frac=0.1, zipf_s=1.3)
    base.update(kw)
    return synth.Workload("fused_small", seed=seed, **base)


@pytest.mark.parametrize("weight_prec", ["mxfp8", "mxfp8_1x32"])
def test_fused_small_against_staged_and_oracle(weight_prec):
    from moe_cases import Case, run_oracle
    w = _small(61)
    rig = Rig(w, weight_prec)
    case = Case(w)
    x = case.x.to(rig.dev)
    ids = torch.from_numpy(case.ids).to(rig.dev)
    sc = torch.from_numpy(case.scores).to(rig.dev)
    base = torch.randn((w.T, w.D), generator=torch.Generator(device=rig.dev).manual_seed(3),
                       device=rig.dev).to(torch.bfloat16)
    staged = rig.run(x, ids, sc, fused=False, out=base.clone(), accumulate=True)
    fused = rig.run(x, ids, sc, fused=True, out=base.clone(), accumulate=True)
    torch.cuda.synchronize()
    assert rig.layer.error_bits() == 0
    _assert_same(fused, staged)
    # the rig's weights came from the device generator: the oracle takes them
    st = omoe.forward(to_f64(case.x), case.ids.astype(np.int64), case.scores, to_f64(rig.w13_bf16),
                      to_f64(rig.w2_bf16), "mxfp8", out_init=to_f64(base),
                      weight_blocks="1x32" if weight_prec == "mxfp8_1x32" else "32x32")
    assert rel_err(to_f64(fused), st["out"]) <= TOL["mxfp8"]
    rig.close()


def test_fused_capped_grid_and_graph_replays():
    """Three CTAs walk every record (each waits on records of the others),
    and a captured graph of the fused forward replays with new inputs."""
    from mixture_experts_routed_route_gb300 import abi
    w = _small(62, T=96, E=12, K=4)
    rig = Rig(w)
    x, ids, sc = rig.inputs(w.T, 62)
    staged = rig.run(x, ids, sc, fused=False)
    abi.moe_ctx_set_max_ctas(rig.layer.ctx, 3)
    capped = rig.run(x, ids, sc, fused=True)
    torch.cuda.synchronize()
    _assert_same(capped, staged)
    abi.moe_ctx_set_max_ctas(rig.layer.ctx, 0)
    # graph: fixed buffers, inputs refreshed between replays
    xg, ig, sg = x.clone(), ids.clone(), sc.clone()
    og = torch.empty_like(staged)
    rig.run(xg, ig, sg, fused=True, out=og)     # warm (kernel set-up outside capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rig.run(xg, ig, sg, fused=True, out=og)
    for seed in (63, 64):
        x2, i2, s2 = rig.inputs(w.T, seed)
        xg.copy_(x2)
        ig.copy_(i2)
        sg.copy_(s2)
        g.replay()
        ref = rig.run(x2, i2, s2, fused=False)
        torch.cuda.synchronize()
        _assert_same(og, ref)
    assert rig.layer.error_bits() == 0
    rig.close()


def test_fused_bad_ids_and_all_inactive():
    from mixture_experts_routed_route_gb300 import abi
    w = _small(65, T=40)
    rig = Rig(w)
    x, ids, sc = rig.inputs(w.T, 65)
    ids[5, 0] = w.E + 3          # counts as inactive and sets the bad-ID bit
    staged = rig.run(x, ids, sc, fused=False)
    torch.cuda.synchronize()
    assert rig.layer.error_bits() & abi.MOE_DEV_ERR_BAD_ID
    fused = rig.run(x, ids, sc, fused=True)
    torch.cuda.synchronize()
    assert rig.layer.error_bits() & abi.MOE_DEV_ERR_BAD_ID
    _assert_same(fused, staged)
    ids.fill_(-1)
    zero = rig.run(x, ids, sc, fused=True)
    torch.cuda.synchronize()
    assert rig.layer.error_bits() == 0
    assert torch.count_nonzero(zero.float()).item() == 0
    rig.close()


def test_fused_wait_runs_out_and_context_stays_usable():
    """With the test stall on, W2 tiles wait for a count nothing reaches: the
    launch returns within a short limit with the timeout bit set, and the
    next launch (stall off) gives the staged result again."""
    from mixture_experts_routed_route_gb300 import abi
    w = _small(66, T=64)
    rig = Rig(w)
    x, ids, sc = rig.inputs(w.T, 66)
    ref = rig.run(x, ids, sc, fused=False)
    torch.cuda.synchronize()
    abi.moe_ctx_test_fused_stall(rig.layer.ctx, 1, 20_000_000)   # about 10 ms per wait
    t0 = time.perf_counter()
    rig.run(x, ids, sc, fused=True)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert rig.layer.error_bits() & abi.MOE_DEV_ERR_TIMEOUT
    assert elapsed < 5.0
    abi.moe_ctx_test_fused_stall(rig.layer.ctx, 0, 0)
    again = rig.run(x, ids, sc, fused=True)
    torch.cuda.synchronize()
    assert rig.layer.error_bits() == 0
    _assert_same(again, ref)
    rig.close()


def test_fused_rejects_what_it_does_not_cover():
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    dev = torch.device("cuda")
    # BF16 context
    w = synth.Workload("fused_bf16", 32, 256, 256, 4, 2, "bf16", "uniform", seed=67)
    w13, w2 = synth.make_weights(w, dev)
    W13, W2 = PreparedWeight(w13, "bf16", with_transpose=False), PreparedWeight(w2, "bf16", with_transpose=False)
    layer = MoELayer(w.T, w.D, w.F, w.E, w.K, "bf16")
    ids, sc = (torch.from_numpy(a).to(dev) for a in synth.make_routing(w))
    x = synth.make_tokens(w, dev)
    out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_forward(layer.ctx, w.T, x, ids, sc, W13.struct, W2.struct, out, None, abi.MOE_FUSED_LAUNCH, None)
    assert ei.value.status == abi.MOE_ERR_UNSUPPORTED
    layer.close()
    # more routes than the single launch takes
    big = _small(68, T=300, K=4)
    rig = Rig(big)
    xb, ib, sb = rig.inputs(big.T, 68)
    with pytest.raises(abi.MoEError) as ei:
        rig.run(xb, ib, sb, fused=True)
    assert ei.value.status == abi.MOE_ERR_UNSUPPORTED
    rig.close()
