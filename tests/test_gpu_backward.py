"""Backward of the CUDA path against the oracle: the dh3 bundles bit-exact
(both sides quantise the same FP32 product s*dY), dX, dW13 and dW2 within the
stated tolerance, zero gradients where no active route reaches."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth
from oracle import formats as fm

from moe_cases import (TOL, Case, check_mx_wgrad, rel_err, run_gpu, run_oracle, saved_blocks, to_f64,
                        unpack_col_sf, unpack_row_sf)

pytestmark = pytest.mark.gpu


def _mx_tiny():
    return synth.Workload("mx_tiny", 128, 256, 256, 8, 2, "mxfp8", "topk_logits", inactive_frac=0.05, seed=31)


def _bf16_skewed():
    return synth.Workload("bf16_skewed", 400, 256, 384, 12, 4, "bf16", "zipf", inactive_frac=0.1, zipf_s=1.4,
                          seed=32)


def _mx_skewed():
    return synth.Workload("mx_skewed", 400, 256, 384, 12, 4, "mxfp8", "zipf", inactive_frac=0.1, zipf_s=1.4,
                          seed=33)


def _mx_d384():
    # D and F not multiples of 256: the store and SwiGLU-backward GEMMs take one weight tile per stage
    return synth.Workload("mx_d384", 200, 384, 384, 8, 3, "mxfp8", "zipf", inactive_frac=0.05, zipf_s=1.2, seed=34)


def _bf16_d384():
    return synth.Workload("bf16_d384", 200, 384, 384, 8, 3, "bf16", "zipf", inactive_frac=0.05, zipf_s=1.2, seed=35)


CASES = {
    "tiny_bf16": lambda: synth.WORKLOADS["tiny_bf16"],
    "bf16_skewed": _bf16_skewed,
    "mx_tiny": _mx_tiny,
    "mx_skewed": _mx_skewed,
    "mx_d384": _mx_d384,
    "bf16_d384": _bf16_d384,
}


@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name):
    case = Case(CASES[name]())
    p = case.w.precision
    g = run_gpu(case)
    o = run_oracle(case)
    assert g["err_bits"] == 0
    for k in ("out", "dx", "dp") if p == "mxfp8" else ("out", "dx", "dp", "dW13", "dW2"):
        assert rel_err(g[k], o[k]) <= TOL[p], k
    assert np.all(g["dp"][case.ids < 0] == 0.0)      # inactive routes get no score gradient
    if p == "mxfp8":
        check_mx_wgrad(g["dW13"], g["dW2"], o["state"], o["grads"])
    dead = np.all(case.ids < 0, axis=1)
    assert np.all(g["dx"][dead] == 0.0)
    # experts that no active route reaches get exact zero weight gradients
    hit = np.zeros(case.w.E, bool)
    hit[case.ids[case.ids >= 0]] = True
    assert np.all(g["dW13"][~hit] == 0.0) and np.all(g["dW2"][~hit] == 0.0)


@pytest.mark.parametrize("name", ["tiny_bf16", "mx_tiny"])
def test_dh3_bundles_bit_exact(name):
    from mixture_experts_routed_route_gb300 import abi
    case = Case(CASES[name]())
    w = case.w
    g = run_gpu(case)
    o = run_oracle(case)
    gr = o["grads"]
    layer = g["layer"]
    rows = int(o["state"]["routing"].poffsets[w.E])
    D, R = w.D, layer.r_cap
    if w.precision == "bf16":
        row = layer.read_buffer(abi.MOE_BUF_DH3ROW, np.uint16, (rows, D))
        np.testing.assert_array_equal(fm.bf16_bits_to_f64(row), gr["dh3_row"])
        col = layer.read_buffer(abi.MOE_BUF_DH3COL, np.uint16, (D, R))[:, :rows]
        np.testing.assert_array_equal(fm.bf16_bits_to_f64(col).T, gr["dh3_col"])
    else:
        blocks = saved_blocks(layer, g["saved"])
        row = layer.read_buffer(abi.MOE_BUF_DH3ROW, np.uint8, (rows, D))
        _, nb_row = abi.moe_ctx_buffer(layer.ctx, abi.MOE_BUF_DH3ROW_SCALE)
        rs = unpack_row_sf(layer.read_buffer(abi.MOE_BUF_DH3ROW_SCALE, np.uint8, (nb_row,)), blocks, rows, D)
        rs = rs.astype(np.int64) - 127
        q, e = fm.mx_quantize(gr["dh3"], axis=-1)
        np.testing.assert_array_equal(fm.e4m3_decode(row), q)
        np.testing.assert_array_equal(rs, e)
        col = layer.read_buffer(abi.MOE_BUF_DH3COL, np.uint8, (D, R))[:, :rows]
        _, nb_col = abi.moe_ctx_buffer(layer.ctx, abi.MOE_BUF_DH3COL_SCALE)
        b_cap = nb_col // ((D // 128) * 512)
        cs = unpack_col_sf(layer.read_buffer(abi.MOE_BUF_DH3COL_SCALE, np.uint8, (nb_col,)), blocks, D, rows, b_cap)
        q, e = fm.mx_quantize(gr["dh3"], axis=0)
        np.testing.assert_array_equal(fm.e4m3_decode(col).T, q)
        np.testing.assert_array_equal(cs.astype(np.int64).T - 127, e)


def test_accumulate_dx_and_fp32_dw():
    case = Case(synth.WORKLOADS["tiny_bf16"])
    init = torch.randn((case.T, case.w.D), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    g = run_gpu(case, dx_init=init.cuda(), dw_fp32=True)
    o = run_oracle(case, dx_init=to_f64(init), dw_fp32=True)
    for k in ("dx", "dW13", "dW2"):
        assert rel_err(g[k], o[k]) <= TOL["bf16"], k


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_all_routes_inactive(precision):
    """Every route ID -1: no expert gets a row, every GEMM has zero tiles, and
    out, dX, dW13, dW2 and the score gradient are exact zeros (the old out /
    dX with the accumulate flags)."""
    w = synth.Workload("all_inactive", 96, 256, 256, 8, 2, precision, "uniform", seed=51)
    ids = np.full((96, 2), -1, np.int32)
    scores = np.zeros((96, 2), np.float32)
    case = Case(w, ids=ids, scores=scores)
    g = run_gpu(case)
    assert g["err_bits"] == 0
    for k in ("out", "dx", "dW13", "dW2", "dp"):
        assert np.all(g[k] == 0.0), k
    o = run_oracle(case)
    assert np.all(o["out"] == 0.0) and np.all(o["dx"] == 0.0)
    init = torch.full((96, w.D), 0.5, dtype=torch.bfloat16)
    ga = run_gpu(case, out_init=init.cuda(), dx_init=init.cuda())
    assert np.all(ga["out"] == 0.5) and np.all(ga["dx"] == 0.5)
