"""Pins of the oracle's NVFP4 format and NVFP4 inference forward ("Dist-MoE:
Speed-of-light distributed Mixture-of-Experts kernels", section 02: E2M1
values with E4M3 block scales and global scales; section 08: NVFP4 inference
with prepared weights), against things other than the oracle itself: the
16 codes and hand-rounded values, hand-worked blocks, a brute-force nearest
search over the E2M1 grid, exact scale invariance, and the routed forward
against the per-token loop and the dense SwiGLU FFN."""

import json
import os

import numpy as np
import pytest

from oracle import formats as fm
from oracle import moe

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "nvfp4_hand_blocks.json")) as f:
        return json.load(f)


def test_e2m1_codes(golden_dir):
    g = _golden(golden_dir)
    vals = fm.e2m1_decode(np.arange(16))
    want = np.array(g["e2m1_values"])
    np.testing.assert_array_equal(vals, want)
    assert np.array_equal(np.signbit(vals), np.signbit(want))     # code 8 is -0
    np.testing.assert_array_equal(fm.e2m1_encode(vals), np.arange(16))
    np.testing.assert_array_equal(fm.round_e2m1(vals), vals)


def test_e2m1_hand_rounding(golden_dir):
    for x, r in _golden(golden_dir)["e2m1_rounding"]:
        got = float(fm.round_e2m1(x))
        assert got == r and np.signbit(got) == np.signbit(r), (x, got, r)


def test_e2m1_rounding_is_the_nearest_grid_point():
    """Brute force: the nearest of the 15 distinct E2M1 values, ties to the
    even code (fraction bit 0), beyond +-6 the largest."""
    grid = np.unique(fm.e2m1_decode(np.arange(16)))
    codes = fm.e2m1_encode(grid)
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-8, 8, 20000), (np.arange(-13, 14) / 2.0 + 0.25),
                        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])])
    d = np.abs(x[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    tie = np.isclose(d, best, rtol=0, atol=0)
    pick = np.where(tie & ((codes & 1) == 0)[None, :], 1, 0) + np.where(tie, 1, 0)
    want = grid[np.argmax(pick, axis=1)]
    np.testing.assert_array_equal(np.abs(fm.round_e2m1(x)), np.abs(want))


def test_nvfp4_hand_rows(golden_dir):
    for r in _golden(golden_dir)["rows"]:
        v = np.array(r["values"], float)[None]
        q, sb, g = fm.nvfp4_quantize(v)
        assert q[0].tolist() == r["q"], r["name"]
        assert sb[0].tolist() == r["block_scales"], r["name"]
        assert float(g[0]) == r["g"], r["name"]
        assert fm.nvfp4_dequantize(q, sb, g)[0].tolist() == r["dequant"], r["name"]


def _fp32_rows(rng, shape, spread=8):
    return (rng.standard_normal(shape) * np.exp2(rng.integers(-spread, spread, shape[:-1] + (1,)))).astype(
        np.float32).astype(np.float64)


def test_nvfp4_scale_invariance():
    """Scaling a row by 2^k scales its global scale by 2^k and leaves every
    code and block scale unchanged (each FP32 step scales exactly)."""
    rng = np.random.default_rng(6)
    v = _fp32_rows(rng, (8, 96))
    q, sb, g = fm.nvfp4_quantize(v)
    for k in (-20, -3, 5, 30):
        q2, sb2, g2 = fm.nvfp4_quantize(v * 2.0 ** k)
        np.testing.assert_array_equal(q2, q)
        np.testing.assert_array_equal(sb2, sb)
        np.testing.assert_array_equal(g2, g * 2.0 ** k)


def test_nvfp4_codes_are_nearest_given_the_block_scale():
    """Given each block's dequantisation factor d = sb g, every code is the
    nearest E2M1 value of v/d (brute force over the grid, ties even), and the
    row's largest block gets the largest E4M3 scale."""
    rng = np.random.default_rng(7)
    v = _fp32_rows(rng, (16, 64))
    q, sb, g = fm.nvfp4_quantize(v)
    grid = np.unique(fm.e2m1_decode(np.arange(16)))
    d = np.repeat((sb * g[:, None]).astype(np.float32).astype(np.float64), 16, axis=1)
    y = (v.astype(np.float32) / d.astype(np.float32)).astype(np.float64)
    dist = np.abs(y[..., None] - grid)
    near = grid[np.argmin(dist, axis=-1)]
    ties = np.sum(dist == dist.min(axis=-1, keepdims=True), axis=-1) > 1
    assert np.all((q == near) | ties)
    blk_amax = np.abs(v).reshape(16, 4, 16).max(axis=-1)
    top = np.argmax(blk_amax, axis=1)
    assert np.all(sb[np.arange(16), top] == 448.0)
    assert np.all(np.abs(q).max(axis=1) == 6.0)


def test_nvfp4_zero_and_inactive():
    v = np.zeros((3, 32))
    v[1, 20] = 3.0
    q, sb, g = fm.nvfp4_quantize(v)
    assert np.all(q[0] == 0) and g[0] == 0 and np.all(sb[0] == 0)
    assert np.all(q[1, :16] == 0) and sb[1, 0] == 0 and q[1, 20] == 6.0


@pytest.mark.parametrize("seed", [0, 1])
def test_nvfp4_routed_forward_matches_per_token_loop(seed):
    rng = np.random.default_rng(40 + seed)
    T, D, F, E, K = 40, 64, 96, 5, 2
    x = rng.standard_normal((T, D)).astype(np.float32).astype(np.float64)
    ids = rng.integers(-1, E, (T, K))
    s = rng.random((T, K)).astype(np.float32)
    w13 = (rng.standard_normal((E, 2 * F, D)) / 8).astype(np.float32).astype(np.float64)
    w2 = (rng.standard_normal((E, D, F)) / 10).astype(np.float32).astype(np.float64)
    st = moe.forward(x, ids, s, w13, w2, "nvfp4")
    pt = moe.forward_per_token(x, ids, s, w13, w2, "nvfp4")
    for t in range(T):
        np.testing.assert_array_equal(st["out"][t], pt[t])


def test_nvfp4_single_expert_is_the_dense_ffn():
    """E=1, K=1, s=1: the dense SwiGLU FFN on NVFP4-quantised operands,
    written out here with the format's dequantised values."""
    rng = np.random.default_rng(44)
    T, D, F = 24, 64, 48
    x = rng.standard_normal((T, D)).astype(np.float32).astype(np.float64)
    w13 = (rng.standard_normal((1, 2 * F, D)) / 8).astype(np.float32).astype(np.float64)
    w2 = (rng.standard_normal((1, D, F)) / 7).astype(np.float32).astype(np.float64)
    out = moe.forward(x, np.zeros((T, 1), int), np.ones((T, 1), np.float32), w13, w2, "nvfp4")["out"]
    xq = fm.nvfp4_fake_quant(x)
    wa = fm.nvfp4_fake_quant(w13[0])
    wb = fm.nvfp4_fake_quant(w2[0])
    h1 = fm.round_bf16(xq @ wa.T)
    g, u = h1[:, :F], h1[:, F:]
    h2 = fm.nvfp4_fake_quant(fm.round_fp32(g / (1 + np.exp(-g)) * u))
    want = fm.round_bf16(fm.round_bf16(h2 @ wb.T))
    np.testing.assert_array_equal(out, want)


def test_nvfp4_has_no_backward():
    rng = np.random.default_rng(45)
    x = rng.standard_normal((8, 32)).astype(np.float32).astype(np.float64)
    w13 = rng.standard_normal((2, 64, 32)).astype(np.float32).astype(np.float64)
    w2 = rng.standard_normal((2, 32, 32)).astype(np.float32).astype(np.float64)
    st = moe.forward(x, np.zeros((8, 1), int), np.ones((8, 1), np.float32), w13, w2, "nvfp4")
    with pytest.raises(AssertionError):
        moe.backward(st, x, w13, w2)
