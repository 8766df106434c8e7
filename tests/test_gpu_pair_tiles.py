"""Grouped GEMMs over row-block pairs (B operands of two consecutive routing
blocks of one expert, up to 256 rows), on one CTA or on CTA pairs (clusters
of two sharing one 256 x 256 MMA), against the same GEMMs over single row
blocks, and against the oracle.

The two tilings contract every output element over the same K order, so the
forward output, the input gradient, both weight gradients and the score
gradient must agree bit for bit.  The cases mix full pairs (256 rows), pairs
whose second block is short, experts with an odd number of blocks (a last
block alone) and experts with a single short block; the SwiGLU forward's
64-feature tiles start on both halves of the weight's 128-row scale atoms
(F = 256, 384).  ("Mixture of Experts: How Routing Becomes GPU
Computation", section 2, "Grouped GEMM": C_e = A_e B_e^T over each expert's
ragged rows; Dist-MoE explainer section 05, "GPU Kernels: Tiles and Warp
Roles": expert row tiles with masked tails.)"""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth

from moe_cases import TOL, Case, check_mx_wgrad, rel_err, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = {
    # 1200 routes over 4 experts, Zipf-skewed: 1 to 5 blocks per expert
    "mx_ragged": lambda: synth.Workload("pair_mx", 600, 256, 256, 4, 2, "mxfp8", "zipf", inactive_frac=0.05,
                                        zipf_s=0.8, seed=81),
    "bf16_ragged": lambda: synth.Workload("pair_bf16", 600, 256, 384, 4, 2, "bf16", "zipf", inactive_frac=0.05,
                                          zipf_s=0.8, seed=82),
    # uniform: every expert about 2 full blocks
    "mx_full": lambda: synth.Workload("pair_full", 512, 512, 384, 4, 2, "mxfp8", "uniform", seed=83),
}

FIELDS = ("out", "dx", "dW13", "dW2", "dp")


def _both(w, **kw):
    case = Case(w)
    a = run_gpu(case, tile_mode=1, **kw)
    b = run_gpu(case, tile_mode=2, **kw)
    for r in (a, b):
        assert r["err_bits"] == 0
    return case, a, b


def _pairs_in(r):
    hdr = r["layer"].saved_field(r["saved"], 0, torch.int32, (16,)).cpu().numpy()
    return int(hdr[1]), int(hdr[4])


@pytest.mark.parametrize("name", list(CASES))
def test_pairs_equal_row_blocks_bitwise(name):
    w = CASES[name]()
    case, a, b = _both(w)
    nblk, npair = _pairs_in(b)
    assert npair < nblk      # some experts do have two or more blocks
    for f in FIELDS:
        np.testing.assert_array_equal(a[f], b[f], err_msg=f)
    o = run_oracle(case)
    tol = TOL[w.precision]
    assert rel_err(b["out"], o["out"]) <= tol
    assert rel_err(b["dx"], o["dx"]) <= tol
    if w.precision == "bf16":
        assert rel_err(b["dW13"], o["dW13"]) <= tol and rel_err(b["dW2"], o["dW2"]) <= tol
    else:
        check_mx_wgrad(b["dW13"], b["dW2"], o["state"], o["grads"])


def test_pairs_mn_major_input_gradient():
    """MXFP8 weights without transposed codes: the W13 input-gradient GEMM
    over pairs reads the forward codes MN-major; same bits as row blocks."""
    w = CASES["mx_full"]()
    case, a, b = _both(w, mn_major=True)
    for f in FIELDS:
        np.testing.assert_array_equal(a[f], b[f], err_msg=f)


def test_pairs_inference_and_clamped_swiglu():
    """Inference (no saved state: h1 and column bundles not written) and the
    clamped SwiGLU with its clip counts, pairs against row blocks."""
    w = CASES["mx_ragged"]()
    case = Case(w)
    res = []
    for mode in (1, 2):
        r = run_gpu(case, training=False, swiglu_limit=0.75, tile_mode=mode)
        assert r["err_bits"] == 0
        res.append((r["out"], r["layer"].clip_stats()))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    assert list(res[0][1]) == list(res[1][1]) and res[0][1][0] > 0


# ---------------------------------------------------------------- CTA pairs
# Mode 3: the forward's pair tiles on clusters of two CTAs, one 256 x 256
# MMA (cta_group::2; block-scaled in MXFP8) per K step over both: each CTA
# holds its own 128 weight rows (SwiGLU: 64 gate + 64 up rows of its own 64
# features) and one routing block of the pair, and drains its own 128
# accumulator lanes; a stage is two 128-element K-chunks.  The contraction
# order per output element is that of the row-block tiles, so the bits must
# match.  The backward's GEMMs keep their usual tiles; a saved state is the
# same whichever tiles wrote it.

CTA_CASES = {
    # D = F = 256: one stage per tile; lone last blocks (the second CTA of the
    # cluster loads no rows) and short second blocks
    "mx_ragged": CASES["mx_ragged"],
    # D = 1024, F = 512: four stages per W13 tile, two per W2 tile (stage ring
    # phases wrap within a tile), two W2 cluster tiles along the features
    "mx_deep": lambda: synth.Workload("pair_deep", 600, 1024, 512, 4, 2, "mxfp8", "zipf", inactive_frac=0.05,
                                      zipf_s=0.8, seed=85),
    # BF16: 128-value stages (eight per W13 tile), two accumulator buffers
    "bf16_deep": lambda: synth.Workload("pair_bf16_deep", 600, 1024, 512, 4, 2, "bf16", "zipf",
                                        inactive_frac=0.05, zipf_s=0.8, seed=86),
}


@pytest.mark.parametrize("max_ctas", [0, 1, 6])
@pytest.mark.parametrize("name", list(CTA_CASES))
def test_cta_pairs_equal_row_blocks_bitwise(name, max_ctas):
    """max_ctas = 6 (three clusters) makes every cluster walk many tiles;
    max_ctas = 1 still launches one cluster of two, which walks them all."""
    w = CTA_CASES[name]()
    case = Case(w)
    a = run_gpu(case, tile_mode=1, max_ctas=max_ctas)
    b = run_gpu(case, tile_mode=3, max_ctas=max_ctas)
    for r in (a, b):
        assert r["err_bits"] == 0
    for f in FIELDS:
        np.testing.assert_array_equal(a[f], b[f], err_msg=f)
    o = run_oracle(case, backward=False)
    assert rel_err(b["out"], o["out"]) <= TOL[w.precision]


def test_cta_pairs_inference_and_clamped_swiglu():
    """Inference through CTA pairs with the clamped SwiGLU: output and clip
    counts equal to row blocks."""
    w = CTA_CASES["mx_deep"]()
    case = Case(w)
    res = []
    for mode in (1, 3):
        r = run_gpu(case, training=False, swiglu_limit=0.75, tile_mode=mode)
        assert r["err_bits"] == 0
        res.append((r["out"], r["layer"].clip_stats()))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    assert list(res[0][1]) == list(res[1][1]) and res[0][1][0] > 0


@pytest.mark.parametrize("prec,D,F", [("mxfp8", 384, 256), ("mxfp8", 512, 384), ("bf16", 384, 256)])
def test_cta_pairs_fall_back_where_k_does_not_divide(prec, D, F):
    """A CTA pair's stage is 256 bytes of K (256 MXFP8 or 128 BF16 values) and
    its W2 tile 256 features: W13 (K = D) and W2 (K = F, 256-feature tiles of
    D) that do not divide take one-CTA pair tiles instead, with the same
    bits (BF16, D = 384: W13 on CTA pairs, W2 not)."""
    w = synth.Workload("pair_fallback", 300, D, F, 3, 2, prec, "uniform", seed=84)
    case = Case(w)
    a = run_gpu(case, training=False, tile_mode=1)
    b = run_gpu(case, training=False, tile_mode=3)
    assert a["err_bits"] == 0 and b["err_bits"] == 0
    np.testing.assert_array_equal(a["out"], b["out"])


def test_cta_pairs_at_the_dense_full_size():
    """The compute-bound diagnostic shape (T=2048, D=7168, F=2048, E=6, K=6,
    every token routed to every expert: 8 full pairs per expert, 28 stages
    per W13 tile, more tiles than clusters).  CTA pairs, forced and by the
    context's default at this density, equal row blocks bit for bit; sampled
    tokens match the oracle (the MXFP8 oracle quantises each token row on its
    own, so a token subset gives the same rows)."""
    from oracle import moe as omoe
    from moe_cases import to_f64
    w = synth.WORKLOADS["e6_dense"]
    case = Case(w)
    a = run_gpu(case, training=False, tile_mode=1)
    b = run_gpu(case, training=False, tile_mode=3)
    c = run_gpu(case, training=False)
    for r in (a, b, c):
        assert r["err_bits"] == 0
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["out"], c["out"])
    tokens = [0, 777, 1500, 2047]
    st = omoe.forward(to_f64(case.x)[tokens], case.ids[tokens].astype(np.int64), case.scores[tokens],
                      to_f64(case.w13), to_f64(case.w2), "mxfp8")
    assert rel_err(b["out"][tokens], st["out"]) <= TOL["mxfp8"]
