"""Activation-slot planner ("Dist-MoE: Speed-of-light distributed
Mixture-of-Experts kernels", section 04 "Activation Packing and Dynamic
Recompute"): the oracle against the worked example the page prints and
brute-force properties; the library's host-side planner (moe_slot_*) and the
input-only saved-state layout against the oracle and the header.  No GPU:
these functions make no CUDA call.
"""

import json
import os

import numpy as np
import pytest

from oracle import slot_plan as sp


@pytest.fixture(scope="module")
def abi():
    from mixture_experts_routed_route_gb300 import build
    if not os.path.exists(os.path.join(build.OUT_DIR, build.LIB_NAME)):
        build.build()
    from mixture_experts_routed_route_gb300 import abi as a
    return a


def _example(golden_dir):
    return json.load(open(os.path.join(golden_dir, "slot_plan_worked_example.json")))


# ------------------------------------------------------------------ oracle pins

def test_oracle_reproduces_the_printed_worked_example(golden_dir):
    ex = _example(golden_dir)
    layers = [(ex["full_bytes"], ex["input_bytes"])] * ex["layers"]
    for preset in ex["presets"]:
        plan = sp.plan_stack(layers, preset["capacity"])
        assert [p["decision"] for p in plan] == preset["decisions"]
        for layer, need in preset["printed_checks"].items():
            assert plan[int(layer)]["need"] == need


def test_oracle_align128():
    assert [sp.align128(n) for n in (0, 1, 127, 128, 129, 8960)] == [0, 128, 128, 128, 256, 8960]


def test_oracle_properties_by_brute_force():
    """Every layer's input fits; a layer keeps only its input exactly when
    its full-state test fails; nothing overlaps or passes the capacity; a slot
    as large as all full states keeps them all; offsets are 128-aligned."""
    rng = np.random.default_rng(5)
    for _ in range(400):
        n = int(rng.integers(1, 9))
        layers = [(int(rng.integers(1, 40)) * 100, int(rng.integers(0, 6)) * 100) for _ in range(n)]
        cap = int(rng.integers(0, sum(sp.align128(f) for f, _ in layers) + 512))
        try:
            plan = sp.plan_stack(layers, cap)
        except MemoryError:
            continue
        end = 0
        for k, (p, (f, i)) in enumerate(zip(plan, layers)):
            assert p["offset"] == end and p["offset"] % 128 == 0
            reserve = sum(sp.align128(i) for _ in range(n - 1 - k))
            fits = p["offset"] + sp.align128(f) + reserve <= cap
            assert (p["decision"] == sp.FULL) == fits
            end += p["bytes"]
        assert end <= cap
    layers = [(1000, 100)] * 5
    assert all(p["decision"] == sp.FULL for p in sp.plan_stack(layers, 5 * 1024))
    # the reserve guarantees the minimum slot: with one input size, a slot
    # holding every layer's input never fails, whatever the full sizes
    for _ in range(300):
        n = int(rng.integers(1, 9))
        i = int(rng.integers(0, 6)) * 100
        layers = [(i + int(rng.integers(0, 40)) * 100, i) for _ in range(n)]   # a full state holds more
        cap = n * sp.align128(i) + int(rng.integers(0, 4000))
        plan = sp.plan_stack(layers, cap)
        if cap < sum(sp.align128(f) for f, _ in layers):
            assert len(plan) == n
        with pytest.raises(MemoryError):
            if n * sp.align128(i) > 0:
                sp.plan_stack(layers, n * sp.align128(i) - 1)
            else:
                raise MemoryError


# ------------------------------------------------------- library vs the oracle

def _lib_plan(abi, layers, cap, max_layers=64):
    slot = abi.moe_slot_init(cap, max_layers)
    out = []
    for k, (f, i) in enumerate(layers):
        out.append(abi.moe_slot_push(slot, f, i, len(layers) - 1 - k))
    return slot, out


def test_library_planner_reproduces_the_worked_example(abi, golden_dir):
    ex = _example(golden_dir)
    layers = [(ex["full_bytes"], ex["input_bytes"])] * ex["layers"]
    for preset in ex["presets"]:
        _, got = _lib_plan(abi, layers, preset["capacity"])
        want = ["full" if fl == 0 else "input" for _, fl in got]
        assert want == preset["decisions"]
        assert all(fl in (0, abi.MOE_SAVE_INPUT_ONLY) for _, fl in got)


def test_library_planner_matches_the_oracle(abi):
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(1, 10))
        layers = [(int(rng.integers(0, 5000)), int(rng.integers(0, 700))) for _ in range(n)]
        cap = int(rng.integers(0, 6000 * n))
        try:
            want = sp.plan_stack(layers, cap)
        except MemoryError:
            with pytest.raises(abi.MoEError) as ei:
                _lib_plan(abi, layers, cap)
            assert ei.value.status == abi.MOE_ERR_CAPACITY
            continue
        slot, got = _lib_plan(abi, layers, cap)
        assert [o for o, _ in got] == [p["offset"] for p in want]
        assert [fl for _, fl in got] == [0 if p["decision"] == sp.FULL else abi.MOE_SAVE_INPUT_ONLY for p in want]
        assert slot.cursor == want[-1]["offset"] + want[-1]["bytes"]
        # backwards in reverse order put the cursor back where each forward found it
        for p in reversed(want):
            abi.moe_slot_pop(slot, p["offset"])
            assert slot.cursor == p["offset"]
        assert slot.layers == 0


def test_library_planner_errors(abi):
    slot = abi.moe_slot_init(10_000, 2)
    a, _ = abi.moe_slot_push(slot, 1000, 100, 0)
    b, _ = abi.moe_slot_push(slot, 1000, 100, 0)
    with pytest.raises(abi.MoEError) as ei:          # max_layers reached
        abi.moe_slot_push(slot, 1000, 100, 0)
    assert ei.value.status == abi.MOE_ERR_CAPACITY
    with pytest.raises(abi.MoEError):                 # not the most recent push
        abi.moe_slot_pop(slot, a)
    abi.moe_slot_pop(slot, b)
    abi.moe_slot_pop(slot, a)
    with pytest.raises(abi.MoEError):                 # empty slot
        abi.moe_slot_pop(slot, 0)
    for bad in ((-1, 100, 0), (1000, -1, 0), (1000, 100, -1)):
        with pytest.raises(abi.MoEError) as ei:
            abi.moe_slot_push(slot, *bad)
        assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    for cap, ml in ((-1, 4), (100, 0), (100, abi.MOE_SLOT_MAX_LAYERS + 1)):
        with pytest.raises(abi.MoEError):
            abi.moe_slot_init(cap, ml)
    with pytest.raises(abi.MoEError) as ei:           # not even the inputs fit
        abi.moe_slot_push(abi.moe_slot_init(1000, 4), 5000, 600, 1)
    assert ei.value.status == abi.MOE_ERR_CAPACITY


# --------------------------------------------------- the input-only state layout

@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
@pytest.mark.parametrize("norm", [False, True])
def test_input_only_layout(abi, precision, norm):
    prec = abi.MOE_BF16 if precision == "bf16" else abi.MOE_MXFP8
    flags = abi.MOE_TRAINING | abi.MOE_REPLAY | (abi.MOE_POST_NORM if norm else 0)
    T, D, F, E, K = 96, 256, 384, 16, 4
    cfg = abi.make_config(T, D, F, E, K, prec, flags)
    routing = (abi.MOE_SAVED_HEADER, abi.MOE_SAVED_COUNTS, abi.MOE_SAVED_OFFSETS, abi.MOE_SAVED_POFFSETS,
               abi.MOE_SAVED_PERM, abi.MOE_SAVED_INV, abi.MOE_SAVED_BLOCKS, abi.MOE_SAVED_SCORES,
               abi.MOE_SAVED_BSTART, abi.MOE_SAVED_ROWBLOCK, abi.MOE_SAVED_PRENORM)
    for f in routing:   # the fields the backward reads from `saved` sit at the same places
        assert abi.moe_saved_input_field(cfg, f) == abi.moe_saved_state_field(cfg, f)
    assert abi.moe_saved_state_field(cfg, abi.MOE_SAVED_PRENORM)[1] == (T * D * 2 if norm else 0)
    for f in (abi.MOE_SAVED_H1, abi.MOE_SAVED_XCOL, abi.MOE_SAVED_XCOL_SCALE, abi.MOE_SAVED_H2COL,
              abi.MOE_SAVED_H2COL_SCALE, abi.MOE_SAVED_H3):
        assert abi.moe_saved_input_field(cfg, f)[1] == 0
        scale = f in (abi.MOE_SAVED_XCOL_SCALE, abi.MOE_SAVED_H2COL_SCALE)
        assert (abi.moe_saved_state_field(cfg, f)[1] > 0) == (precision == "mxfp8" or not scale)
    off, nb = abi.moe_saved_input_field(cfg, abi.MOE_SAVED_X)
    assert nb == T * D * 2 and off % 256 == 0
    assert abi.moe_saved_state_field(cfg, abi.MOE_SAVED_X)[1] == 0
    total = abi.moe_saved_input_bytes(cfg)
    assert off + nb <= total < off + nb + 256
    # the point of it: a small fraction of the full state
    assert total < abi.moe_saved_state_bytes(cfg) / 4


def test_replay_needs_a_training_context(abi):
    import ctypes
    cfg = abi.make_config(64, 256, 256, 8, 2, abi.MOE_BF16, abi.MOE_REPLAY)
    ctx = ctypes.c_void_p()
    # rejected on the host before any CUDA call
    assert abi.LIB.moe_ctx_create(ctypes.byref(cfg), ctypes.byref(ctx)) == abi.MOE_ERR_INVALID_ARG


def test_activation_slot_wrapper_on_a_host_buffer(abi):
    """layer.ActivationSlot: views at the planner's offsets, sized for the
    decision, given back in reverse order (a CPU buffer stands in for HBM)."""
    import types
    import torch
    from mixture_experts_routed_route_gb300.layer import ActivationSlot
    cfg = abi.make_config(64, 256, 256, 8, 2, abi.MOE_MXFP8, abi.MOE_TRAINING | abi.MOE_REPLAY)
    layer = types.SimpleNamespace(cfg=cfg)
    full, inp = abi.moe_saved_state_bytes(cfg), abi.moe_saved_input_bytes(cfg)
    cap = sp.align128(full) * 2 + sp.align128(inp) * 2
    slot = ActivationSlot(cap, max_layers=4, device="cpu")
    want = sp.plan_stack([(full, inp)] * 4, cap)
    got = [slot.push(layer, 3 - l) for l in range(4)]
    base = slot.buf.data_ptr()
    for (view, input_only), p in zip(got, want):
        assert input_only == (p["decision"] == sp.INPUT)
        assert view.data_ptr() - base == p["offset"]
        assert view.numel() == (inp if input_only else full)
    assert [d for _, d in got] == [False, False, True, True]
    with pytest.raises(abi.MoEError):
        slot.pop(got[0][0])            # not the most recent
    for view, _ in reversed(got):
        slot.pop(view)
    assert slot.slot.layers == 0 and slot.slot.cursor == 0
