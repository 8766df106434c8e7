"""The C-ABI library loads and exports every function include/*.h declare
(the boundary, moe_gb300.h, and the test inspection calls,
moe_gb300_testing.h), and the binding's structs match the header (no GPU needed: no
compute call is made)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")
TESTING_HEADER = os.path.join(ROOT, "include", "moe_gb300_testing.h")


def _declared_functions():
    names = []
    for inc in os.listdir(os.path.join(ROOT, "include")):
        if not inc.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", inc)).read()
        names += re.findall(r"^MOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_routed_route_gb300 import build
    path = os.path.join(build.OUT_DIR, build.LIB_NAME)
    if not os.path.exists(path):
        build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = set(_declared_functions())
    for required in ("moe_ctx_create", "moe_ctx_destroy", "moe_forward", "moe_backward",
                     "prepare_block_scaled_weight", "moe_saved_state_bytes", "moe_ctx_get_error"):
        assert required in names


def test_product_header_holds_no_test_inspection_calls():
    """Scratch inspection and host copies live in the testing header only."""
    text = open(HEADER).read()
    for name in ("moe_debug_copy_to_host", "moe_ctx_buffer", "MOE_BUF_XROW"):
        assert name not in text, name
    testing = open(TESTING_HEADER).read()
    assert "moe_debug_copy_to_host" in testing and "moe_ctx_buffer" in testing


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol(lib):
    from mixture_experts_routed_route_gb300 import abi
    for name in _declared_functions():
        assert name in abi._SIGNATURES, name
        assert callable(getattr(abi, name)), name


def test_struct_layouts_match_header():
    from mixture_experts_routed_route_gb300 import abi
    assert ctypes.sizeof(abi.moe_config) == 8 * 4
    assert ctypes.sizeof(abi.moe_weight) == 16 + 4 * 8
    assert abi.moe_weight.data.offset == 16
    assert ctypes.sizeof(abi.moe_slot) == 8 + 8 + 4 + 4 + abi.MOE_SLOT_MAX_LAYERS * (8 + 4)
    assert abi.moe_slot.offset.offset == 24


def test_host_side_sizes_without_gpu(lib):
    """Pure host calls: capacity and layout arithmetic."""
    from mixture_experts_routed_route_gb300 import abi
    cfg = abi.make_config(2048, 7168, 2048, 384, 6, abi.MOE_MXFP8, abi.MOE_TRAINING)
    r = abi.moe_row_capacity(cfg)
    assert r % 128 == 0 and r >= 2048 * 6 + 31 * 384 + 128
    sb = abi.moe_saved_state_bytes(cfg)
    spans = []
    for f in range(abi.MOE_SAVED_NUM_FIELDS):
        off, nb = abi.moe_saved_state_field(cfg, f)
        assert off % 256 == 0 and off + nb <= sb
        spans.append((off, off + nb))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))     # fields do not overlap
    # routing fields come first, then h1 and the column bundles
    routing = [abi.moe_saved_state_field(cfg, f)[0] for f in (abi.MOE_SAVED_BSTART, abi.MOE_SAVED_ROWBLOCK)]
    assert max(routing) < abi.moe_saved_state_field(cfg, abi.MOE_SAVED_H1)[0]
    assert abi.moe_saved_state_field(cfg, abi.MOE_SAVED_H1)[1] == r * 2 * 2048 * 2
    bad = abi.make_config(2048, 7168, 2048, 2000, 6, abi.MOE_MXFP8, 0)
    assert abi.moe_row_capacity(bad) == 0 and abi.moe_saved_state_bytes(bad) == 0
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_ctx_create(bad)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    # the clamp limit must be finite and non-negative
    for lim in (float("nan"), -1.0, float("inf")):
        assert abi.moe_row_capacity(abi.make_config(2048, 7168, 2048, 384, 6, abi.MOE_MXFP8, 0, lim)) == 0
    assert abi.moe_row_capacity(abi.make_config(2048, 7168, 2048, 384, 6, abi.MOE_MXFP8, 0, 7.0)) == r
    odd = abi.make_config(64, 200, 256, 8, 2, abi.MOE_BF16, 0)
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_ctx_create(odd)
    assert ei.value.status in (abi.MOE_ERR_INVALID_ARG, abi.MOE_ERR_UNSUPPORTED)


def test_context_setters_reject_null_context(lib):
    """Host-side argument checks that need no device."""
    from mixture_experts_routed_route_gb300 import abi
    assert abi.LIB.moe_ctx_set_max_ctas(None, 4) == abi.MOE_ERR_INVALID_ARG
    assert abi.LIB.moe_ctx_enable_stage_timing(None, 1) == abi.MOE_ERR_INVALID_ARG


def test_weight_bytes_without_gpu(lib):
    from mixture_experts_routed_route_gb300 import abi
    E, N, K = 6, 256, 384
    atoms = (E * N // 128) * (K // 128) * 512            # one 512-byte atom per 128 x 128 block
    assert abi.moe_weight_bytes(abi.MOE_MXFP8, E, N, K, True) == (E * N * K, atoms + 16, E * K * N, atoms + 16)
    assert abi.moe_weight_bytes(abi.MOE_MXFP8, E, N, K, False) == (E * N * K, atoms + 16, 0, 0)
    assert abi.moe_weight_bytes(abi.MOE_MXFP8_1X32, E, N, K, False) == (E * N * K, atoms + 16, 0, 0)
    # 2: the input-gradient scales only (MN-major input-gradient GEMMs)
    assert abi.moe_weight_bytes(abi.MOE_MXFP8, E, N, K, 2) == (E * N * K, atoms + 16, 0, atoms + 16)
    assert abi.moe_weight_bytes(abi.MOE_BF16, E, 96, 64, True) == (E * 96 * 64 * 2, 0, E * 64 * 96 * 2, 0)
    for bad in ((abi.MOE_MXFP8, E, 96, K, True),        # MXFP8 tiles N and K by 128
                (abi.MOE_MXFP8_1X32, E, N, K, True),    # inference weights have no transpose
                (abi.MOE_BF16, 0, 64, 64, True),
                (abi.MOE_BF16, E, 48, 64, True),
                (abi.MOE_BF16, E, 96, 64, 2),           # BF16 has no scales-only orientation
                (abi.MOE_MXFP8, E, N, K, 3),
                (7, E, N, K, False)):
        with pytest.raises(abi.MoEError) as ei:
            abi.moe_weight_bytes(*bad)
        assert ei.value.status == abi.MOE_ERR_INVALID_ARG


def test_nvfp4_host_side_checks_without_gpu(lib):
    """NVFP4: weight sizes (codes and block scales 9/16 byte per value, one
    FP32 scale per row), an inference-only context, no transposed weights."""
    from mixture_experts_routed_route_gb300 import abi
    E, N, K = 6, 256, 384
    assert abi.moe_weight_bytes(abi.MOE_NVFP4, E, N, K, False) == (E * N * K * 9 // 16, E * N * 4, 0, 0)
    assert abi.moe_weight_bytes(abi.MOE_NVFP4, 1, 128, 64, False) == (4608, 512, 0, 0)   # one chunk
    for bad in ((abi.MOE_NVFP4, E, N, K, True),         # no backward orientation
                (abi.MOE_NVFP4, E, 96, K, False),       # 128-row chunks
                (abi.MOE_NVFP4, E, N, 96, False)):      # 64-value chunks
        with pytest.raises(abi.MoEError) as ei:
            abi.moe_weight_bytes(*bad)
        assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    cfg = abi.make_config(2048, 7168, 2048, 384, 6, abi.MOE_NVFP4, 0)
    assert abi.moe_row_capacity(cfg) > 0 and abi.moe_ctx_scratch_bytes(cfg) > 0
    for flags in (abi.MOE_TRAINING, abi.MOE_TRAINING | abi.MOE_REPLAY, abi.MOE_POST_NORM):
        with pytest.raises(abi.MoEError) as ei:
            abi.moe_ctx_create(abi.make_config(2048, 7168, 2048, 384, 6, abi.MOE_NVFP4, flags))
        assert ei.value.status == abi.MOE_ERR_UNSUPPORTED
    # transposed outputs are rejected before any device work
    fake = ctypes.c_void_p(256)
    st = abi.LIB.prepare_block_scaled_weight(fake, E, N, K, abi.MOE_NVFP4, fake, fake, fake, None, None)
    assert st == abi.MOE_ERR_INVALID_ARG


def test_binding_constants_match_the_header():
    """Every #define and enum value of the header that the binding restates
    has the same value there (the binding is written by hand)."""
    from mixture_experts_routed_route_gb300 import abi
    text = open(HEADER).read() + open(TESTING_HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    values = {}
    for name, val in re.findall(r"^#define\s+(MOE_[A-Z0-9_]+)\s+\(?([0-9xa-fA-F]+)(?:u|ull)?", text, flags=re.M):
        values[name] = int(val, 0)
    for m in re.finditer(r"^#define\s+(MOE_[A-Z0-9_]+)\s+\(([0-9]+)ull\s*<<\s*([0-9]+)\)", text, flags=re.M):
        values[m.group(1)] = int(m.group(2)) << int(m.group(3))
    for body in re.findall(r"typedef enum\s*\{(.*?)\}", text, flags=re.S):
        for name, val in re.findall(r"(MOE_[A-Z0-9_]+)\s*=\s*([0-9]+)", body):
            values[name] = int(val)
    checked = 0
    for name, val in values.items():
        if hasattr(abi, name):
            assert getattr(abi, name) == val, name
            checked += 1
    assert checked >= 60
    for required in ("MOE_REPLAY", "MOE_SAVE_INPUT_ONLY", "MOE_REPLAY_FORWARD", "MOE_SAVED_X", "MOE_BUF_REPLAY",
                     "MOE_SLOT_MAX_LAYERS", "MOE_SAVED_NUM_FIELDS", "MOE_BUF_NUM", "MOE_STATIC_SCRATCH_BYTES"):
        assert required in values and hasattr(abi, required), required
