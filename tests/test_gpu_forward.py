"""Forward of the CUDA path against the oracle, stage by stage: the gathered
(and MXFP8-quantised) rows bit-exact, the prepared weights bit-exact, h1
within the FP32-accumulation bound of the exact product of the same
quantised operands, and h3 / out within the stated tolerance."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth
from oracle import formats as fm
from oracle import moe as omoe

from moe_cases import (TOL, Case, rel_err, run_gpu, run_oracle, saved_blocks, to_f64, unpack_col_sf, unpack_row_sf,
                        unpack_weight_sf)

pytestmark = pytest.mark.gpu


def _mx_tiny():
    return synth.Workload("mx_tiny", 128, 256, 256, 8, 2, "mxfp8", "topk_logits", inactive_frac=0.05, seed=21)


def _bf16_skewed():
    return synth.Workload("bf16_skewed", 400, 256, 384, 12, 4, "bf16", "zipf", inactive_frac=0.1, zipf_s=1.4,
                          seed=22)


def _mx_skewed():
    return synth.Workload("mx_skewed", 400, 256, 384, 12, 4, "mxfp8", "zipf", inactive_frac=0.1, zipf_s=1.4,
                          seed=23)


CASES = {
    "tiny_bf16": lambda: synth.WORKLOADS["tiny_bf16"],
    "bf16_skewed": _bf16_skewed,
    "mx_tiny": _mx_tiny,
    "mx_skewed": _mx_skewed,
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_matches_oracle(name):
    case = Case(CASES[name]())
    p = case.w.precision
    g = run_gpu(case, backward=False)
    o = run_oracle(case, backward=False)
    assert g["err_bits"] == 0
    assert rel_err(g["out"], o["out"]) <= TOL[p]
    # tokens whose routes are all inactive produce exact zeros
    dead = np.all(case.ids < 0, axis=1)
    assert np.all(g["out"][dead] == 0.0)


@pytest.mark.parametrize("name", list(CASES))
def test_forward_stages(name):
    from mixture_experts_routed_route_gb300 import abi
    case = Case(CASES[name]())
    w = case.w
    p = w.precision
    g = run_gpu(case, backward=False)
    st = run_oracle(case, backward=False)["state"]
    layer = g["layer"]
    rows = int(st["routing"].poffsets[w.E])
    D, F = w.D, w.F
    if p == "bf16":
        xr = layer.read_buffer(abi.MOE_BUF_XROW, np.uint16, (rows, D))
        np.testing.assert_array_equal(fm.bf16_bits_to_f64(xr), st["xq"])
    else:
        xr = layer.read_buffer(abi.MOE_BUF_XROW, np.uint8, (rows, D))
        _, nbytes = abi.moe_ctx_buffer(layer.ctx, abi.MOE_BUF_XROW_SCALE)
        atoms = layer.read_buffer(abi.MOE_BUF_XROW_SCALE, np.uint8, (nbytes,))
        xs = unpack_row_sf(atoms, saved_blocks(layer, g["saved"]), rows, D)
        q, e = fm.mx_quantize(st["xg"], axis=-1)
        np.testing.assert_array_equal(fm.e4m3_decode(xr), q)
        np.testing.assert_array_equal(xs.astype(np.int64) - 127, e)
        # the column bundle the same pass writes (the W13 weight gradient's
        # operand): 32-row blocks from each expert's first row
        sv = g["saved"].cpu().numpy()
        off, nb = abi.moe_saved_state_field(layer.cfg, abi.MOE_SAVED_XCOL)
        xc = sv[off:off + D * layer.r_cap].reshape(D, layer.r_cap)[:, :rows]
        off, nb = abi.moe_saved_state_field(layer.cfg, abi.MOE_SAVED_XCOL_SCALE)
        b_cap = nb // ((D // 128) * 512)
        cs = unpack_col_sf(sv[off:off + nb], saved_blocks(layer, g["saved"]), D, rows, b_cap)
        q, e = fm.mx_quantize(st["xg"], axis=0)
        np.testing.assert_array_equal(fm.e4m3_decode(xc).T, q)
        np.testing.assert_array_equal(cs.astype(np.int64).T - 127, e)
    # h1 (saved, BF16) within half a BF16 ulp plus the FP32 accumulation bound
    # of the exact product of the same quantised operands
    h1 = layer.saved_field(g["saved"], abi.MOE_SAVED_H1, torch.bfloat16, (layer.r_cap, 2 * F))
    h1 = to_f64(h1[:rows])
    w13 = to_f64(case.w13)
    exact = np.zeros((rows, 2 * F))
    absdot = np.zeros((rows, 2 * F))
    rt = st["routing"]
    for e in range(w.E):
        a, b = rt.poffsets[e], rt.poffsets[e + 1]
        if a == b:
            continue
        we = omoe.prepare_weight(w13[e], p)
        exact[a:b] = st["xq"][a:b] @ we.T
        absdot[a:b] = np.abs(st["xq"][a:b]) @ np.abs(we).T
    bound = np.abs(exact) * 2.0 ** -8 + absdot * D * 2.0 ** -23
    assert np.all(np.abs(h1 - exact) <= bound)
    # h3 per padded row (a training forward keeps it in the saved state)
    h3 = layer.saved_field(g["saved"], abi.MOE_SAVED_H3, torch.bfloat16, (layer.r_cap, D))
    assert rel_err(to_f64(h3[:rows]), st["h3"]) <= TOL[p]


def test_accumulate_out_adds_shared_expert_first():
    case = Case(synth.WORKLOADS["tiny_bf16"])
    init = torch.randn((case.T, case.w.D), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    g = run_gpu(case, backward=False, out_init=init.cuda())
    o = run_oracle(case, backward=False, out_init=to_f64(init))
    assert rel_err(g["out"], o["out"]) <= TOL["bf16"]


def test_weight_prep_mx_bit_exact():
    from mixture_experts_routed_route_gb300.layer import PreparedWeight
    w = synth.Workload("wprep", 1, 256, 128, 3, 1, "mxfp8", "uniform", seed=24)
    w13, _ = synth.make_weights(w, "cpu")
    w13[1, 5, 70] = 300.0          # an outlier in one 32x32 tile
    pw = PreparedWeight(w13.cuda(), "mxfp8", with_transpose=True)
    q, e = fm.mx_quantize_weight_32x32(to_f64(w13))
    E, N, K = w13.shape
    np.testing.assert_array_equal(fm.e4m3_decode(pw.data.cpu().numpy()), q)
    sf = unpack_weight_sf(pw.scale.cpu().numpy(), E * N, K).reshape(E, N, K // 32).astype(np.int64) - 127
    np.testing.assert_array_equal(sf, np.repeat(e, 32, axis=1))
    np.testing.assert_array_equal(fm.e4m3_decode(pw.data_t.cpu().numpy()), np.swapaxes(q, 1, 2))
    sft = unpack_weight_sf(pw.scale_t.cpu().numpy(), E * K, N).reshape(E, K, N // 32).astype(np.int64) - 127
    np.testing.assert_array_equal(sft, np.repeat(np.swapaxes(e, 1, 2), 32, axis=1))


def test_weight_prep_bf16_transpose():
    from mixture_experts_routed_route_gb300.layer import PreparedWeight
    w = synth.Workload("wprep", 1, 256, 128, 2, 1, "bf16", "uniform", seed=25)
    w13, _ = synth.make_weights(w, "cpu")
    pw = PreparedWeight(w13.cuda(), "bf16", with_transpose=True)
    assert torch.equal(pw.data_t.cpu(), w13.transpose(1, 2).contiguous())


def test_zero_tokens_is_a_no_op():
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    w = synth.WORKLOADS["tiny_bf16"]
    layer = MoELayer(16, w.D, w.F, w.E, w.K, "bf16")
    w13, w2 = synth.make_weights(w, "cuda")
    W13, W2 = PreparedWeight(w13, "bf16", False), PreparedWeight(w2, "bf16", False)
    x = torch.empty((0, w.D), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((0, w.K), dtype=torch.int32, device="cuda")
    sc = torch.empty((0, w.K), dtype=torch.float32, device="cuda")
    out = torch.empty((0, w.D), dtype=torch.bfloat16, device="cuda")
    abi.moe_forward(layer.ctx, 0, None, None, None, W13.struct, W2.struct, None)
    layer.forward(x, ids, sc, W13, W2, out=out)
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_forward(layer.ctx, 17, x, ids, sc, W13.struct, W2.struct, out)
    assert ei.value.status == abi.MOE_ERR_CAPACITY
    assert layer.error_bits() == 0


def test_stage_timing_graph_survives_disable():
    """A graph captured with stage timing on keeps recording into the
    context's events after timing is disabled (they live until the context
    is destroyed), so it can be replayed and its stage times read."""
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    w = synth.WORKLOADS["tiny_bf16"]
    case = Case(w)
    dev = torch.device("cuda")
    layer = MoELayer(w.T, w.D, w.F, w.E, w.K, "bf16")
    W13 = PreparedWeight(case.w13.to(dev), "bf16", with_transpose=False)
    W2 = PreparedWeight(case.w2.to(dev), "bf16", with_transpose=False)
    x = case.x.to(dev)
    ids = torch.from_numpy(case.ids).to(dev)
    sc = torch.from_numpy(case.scores).to(dev)
    out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
    layer.forward(x, ids, sc, W13, W2, out=out)        # eager once (kernel attributes)
    torch.cuda.synchronize()
    abi.moe_ctx_enable_stage_timing(layer.ctx, True)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x, ids, sc, W13, W2, out=out)
    abi.moe_ctx_enable_stage_timing(layer.ctx, False)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        times = abi.moe_ctx_stage_times(layer.ctx, 0)
        assert len(times) == abi.MOE_FWD_STAGES and all(t >= 0 for t in times)
    del graph
    layer.close()
