"""Host-side accounting of bench.py (no GPU): the algorithmic bytes a stage
is charged and the oracle sample's bounds."""

import numpy as np

import bench
from mixture_experts_routed_route_gb300 import synth


def test_gemm_weight_bytes_count_only_routed_experts():
    w = synth.WORKLOADS["e384_mxfp8_zipf_train"]
    q = 1 + 1 / 32
    Rp, R = 20000, 11059
    full_f, full_b = bench.stage_bytes(w, Rp, R, w.precision, True)
    used_f, used_b = bench.stage_bytes(w, Rp, R, w.precision, True, experts_used=381)
    D, F = w.D, w.F
    # the weight-streaming GEMMs lose exactly the three idle experts' weights
    assert full_f["gemm_w13_swiglu"] - used_f["gemm_w13_swiglu"] == 3 * 2 * F * D * q
    assert full_f["gemm_w2"] - used_f["gemm_w2"] == 3 * D * F * q
    assert full_b["gemm_w13_dgrad"] - used_b["gemm_w13_dgrad"] == 3 * 2 * F * D * q
    assert full_b["gemm_w2_dgrad_swiglu_bwd"] - used_b["gemm_w2_dgrad_swiglu_bwd"] == 3 * D * F * q
    # the weight gradients still write every expert's dW (zeros for idle ones)
    assert used_b["gemm_w13_wgrad"] == full_b["gemm_w13_wgrad"]
    assert used_b["gemm_w2_wgrad"] == full_b["gemm_w2_wgrad"]
    assert used_b["gemm_w13_wgrad"] >= w.E * 2 * F * D * 2


def test_one_token_step_charges_six_experts():
    w = synth.WORKLOADS["decode_e384_t1"]
    ids, _ = synth.make_routing(w)
    used = int(np.unique(np.asarray(ids)[np.asarray(ids) >= 0]).size)
    assert used == w.K == 6
    f, _ = bench.stage_bytes(w, 32 * used, used, w.precision, False, experts_used=used)
    assert f["gemm_w13_swiglu"] < 0.2e9 and f["gemm_w2"] < 0.1e9


def test_sample_experts_are_a_nested_seeded_prefix():
    w = synth.WORKLOADS["e384_mxfp8_zipf_train"]
    ids, _ = synth.make_routing(w)
    a = bench.pick_sample_experts(w, ids, 6)
    b = bench.pick_sample_experts(w, ids, 16)
    assert b[:6] == a and len(set(b)) == 16
    present = set(int(e) for e in np.asarray(ids).reshape(-1) if e >= 0)
    assert set(b) <= present


def test_accumulated_fp32_weight_gradients_count_a_read_and_a_write():
    w = synth.WORKLOADS["ten_layer_graph"]
    Rp, R = 40000, 32768
    _, bf = bench.stage_bytes(w, Rp, R, w.precision, True)
    _, acc = bench.stage_bytes(w, Rp, R, w.precision, True, dw_bytes=8)
    D, F, E = w.D, w.F, w.E
    assert acc["gemm_w13_wgrad"] - bf["gemm_w13_wgrad"] == E * 2 * F * D * (8 - 2)
    assert acc["gemm_w2_wgrad"] - bf["gemm_w2_wgrad"] == E * D * F * (8 - 2)
    for k in bf:     # nothing else depends on the weight-gradient format
        if "wgrad" not in k:
            assert acc[k] == bf[k]


def test_gemm_flops_add_up_to_the_step():
    """The per-GEMM useful FLOPs sum to the step's: 6 R D F forward (W13 is
    2F wide, W2 F deep), 12 R D F more for the four backward GEMMs."""
    fwd = bench.GEMM_FLOPS["gemm_w13_swiglu"] + bench.GEMM_FLOPS["gemm_w2"]
    assert fwd == 6.0
    assert sum(bench.GEMM_FLOPS.values()) == 18.0
    w = synth.WORKLOADS["e6_dense"]
    R = w.T * w.K
    ms = {"route": 0.02, "gemm_w13_swiglu": 0.3, "gemm_w2": 0.15, "combine": 0.04}
    g = bench.gemm_tensor(ms, R, w, 1000.0)
    want = 6.0 * R * w.D * w.F / 0.45e-3 / 1e12
    assert abs(g["tflops"] - want) < 0.1 and abs(g["tensor_frac"] - want / 1000.0) < 1e-4
    assert set(g["per_gemm_tensor_frac"]) == {"gemm_w13_swiglu", "gemm_w2"}
    assert bench.gemm_tensor({"route": 0.02}, R, w, 1000.0) is None


def test_roofline_bound_follows_arithmetic_intensity():
    """The dominant kernel is reported under the tensor roof when its useful
    FLOPs per algorithmic byte exceed the ridge (peak FLOP/s over copy
    bandwidth), else under HBM: the dense E=6 W13 (about 2400 FLOP/B) is
    tensor-bound, the E=384 training step's W13 weight gradient (about 28) is
    bound by its dW bytes."""
    pk = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "measured"}
    peak8 = 2 * pk["bf16_tflops"]
    w = synth.WORKLOADS["e6_dense"]
    R = w.T * w.K
    fb, _ = bench.stage_bytes(w, R, R, w.precision, False)
    r = bench.roofline("gemm_w13_swiglu", 0.25, fb["gemm_w13_swiglu"], R, w, pk, peak8, None)
    flops = 4.0 * R * w.D * w.F
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - flops / 0.25e-3 / 1e12) < 0.1 and abs(r["frac"] - r["achieved"] / peak8) < 1e-4
    assert r["flop_per_byte"] > r["ridge_flop_per_byte"]
    w4 = synth.WORKLOADS["e384_mxfp8_zipf_train"]
    _, bb = bench.stage_bytes(w4, 20000, 11059, w4.precision, True)
    r4 = bench.roofline("gemm_w13_wgrad", 3.5, bb["gemm_w13_wgrad"], 11059, w4, pk, peak8, 123)
    assert r4["bound"] == "hbm" and r4["unit"] == "GB/s" and r4["traffic"] == 123
    assert abs(r4["achieved"] - bb["gemm_w13_wgrad"] / 3.5e-3 / 1e9) < 0.1
    # a stage with no GEMM FLOPs (routing, gathers, combine) is always HBM
    assert bench.roofline("combine", 0.04, 1e8, R, w, pk, peak8, None)["bound"] == "hbm"
