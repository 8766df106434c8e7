"""Pins of the fp64 oracle against things other than itself.

Each test ties one oracle function to a closed form, a library routine, a
value the pages print, brute force, or finite differences, chosen so that a
plausible slip (a dropped term, a wrong sign or index, a transposed operand,
an off-by-one scale exponent) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as fm
from oracle import moe

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ formats

def test_bf16_rounding_matches_torch_cast():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, -3.3e-39]]).astype(np.float32)
    ours = fm.round_bf16(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_fp32_rounding_matches_numpy_cast():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000)
    np.testing.assert_array_equal(fm.round_fp32(v), v.astype(np.float32).astype(np.float64))


def test_e4m3_all_codes_round_trip():
    codes = np.arange(256, dtype=np.uint8)
    vals = fm.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254          # 0x7F and 0xFF are NaN
    assert np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0
    assert vals[1] == 2.0 ** -9         # smallest subnormal
    np.testing.assert_array_equal(fm.round_e4m3(vals[finite]), vals[finite])
    back = fm.e4m3_encode(vals[finite])
    # +0 and -0 are distinct codes with equal value; compare values for those
    np.testing.assert_array_equal(fm.e4m3_decode(back), vals[finite])
    np.testing.assert_array_equal(back[codes[finite] != 0x80], codes[finite][codes[finite] != 0x80])


def test_e4m3_rounding_matches_torch_cast_in_range():
    rng = np.random.default_rng(2)
    v = rng.uniform(-464, 464, 50000) * 2.0 ** rng.integers(-14, 1, 50000)
    v = v.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(fm.round_e4m3(v), ref)


def test_e4m3_hand_cases(golden_dir):
    for c in _load(golden_dir, "e4m3_hand_cases.json")["cases"]:
        r = float(fm.round_e4m3(c["value"]))
        assert r == c["rounded"], c
        assert int(fm.e4m3_encode(r)) == c["code"], c


def test_e8m0_decode():
    assert fm.e8m0_decode(127) == 1.0
    assert fm.e8m0_decode(0) == 2.0 ** -127
    assert fm.e8m0_decode(254) == 2.0 ** 127
    assert np.isnan(fm.e8m0_decode(255))


def test_mx_hand_blocks(golden_dir):
    for b in _load(golden_dir, "mx_hand_blocks.json")["blocks"]:
        v = np.full(32, b["fill"])
        for i, x in b["set"].items():
            v[int(i)] = x
        q, e = fm.mx_quantize(v[None, :])
        assert int(e[0, 0]) + 127 == b["scale_byte"], b["name"]
        qx = np.full(32, b["q_fill"])
        for i, x in b["q_set"].items():
            qx[int(i)] = x
        np.testing.assert_array_equal(q[0], qx, err_msg=b["name"])
        d = np.full(32, b["deq_fill"])
        for i, x in b["deq_set"].items():
            d[int(i)] = x
        np.testing.assert_array_equal(fm.mx_dequantize(q, e)[0], d, err_msg=b["name"])


def test_mx_axis_and_block_alignment():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((64, 96)) * np.exp(rng.standard_normal((64, 96)))
    # along rows: blocks are rows [0,32) and [32,64), quantised independently
    full = fm.mx_fake_quant(v, axis=0)
    top = fm.mx_fake_quant(v[:32], axis=0)
    np.testing.assert_array_equal(full[:32], top)
    # along rows == along columns of the transpose
    np.testing.assert_array_equal(full, fm.mx_fake_quant(v.T, axis=-1).T)
    # elements in E4M3's normal range lie within half an ulp (2^-4 relative)
    # of v; elements scaled past 448 saturate (the OCP rule lets the block
    # maximum land in [256, 512))
    q, e = fm.mx_quantize(v, axis=0)
    y = v * np.repeat(np.ldexp(1.0, -e), 32, axis=0)
    normal = (np.abs(y) >= 2.0 ** -6) & (np.abs(y) < 448)
    rel = np.abs(full - v) / np.abs(v)
    assert np.all(rel[normal] <= 2.0 ** -4 + 1e-12)
    sat = np.abs(y) >= 464
    assert np.all(np.abs(q[sat]) == 448.0)
    assert np.all(np.sign(full[full != 0]) == np.sign(v[full != 0]))


def test_mx_weight_32x32_single_scale_per_tile():
    rng = np.random.default_rng(4)
    w = rng.standard_normal((2, 64, 96))
    w[0, 5, 70] = 1000.0
    q, e = fm.mx_quantize_weight_32x32(w)
    assert e.shape == (2, 2, 3)
    assert e[0, 0, 2] == int(math.floor(math.log2(1000.0))) - 8
    # the tile's one scale equals the row-wise scale of the tile's whole content
    tile = w[0, 0:32, 64:96].reshape(1, -1)[:, :32 * 32]
    amax = np.abs(tile).max()
    assert e[0, 0, 2] == fm.mx_shared_exponent(amax)
    # same exponent drives the transpose: quantising w^T with the tile rule gives q^T
    qT, eT = fm.mx_quantize_weight_32x32(np.swapaxes(w, 1, 2))
    np.testing.assert_array_equal(qT, np.swapaxes(q, 1, 2))
    np.testing.assert_array_equal(eT, np.swapaxes(e, 1, 2))


def _tile_scaled_weight(E=2, NT=3, KT=5, seed=9):
    """Weights [E, 32 NT, 32 KT] whose tile (i, j) of expert x holds values
    in [-1, 1] with one element exactly 1, times 2^(3i - 5j + x): every tile
    has its own power-of-two scale, and the known maximum fixes its
    exponent 3i - 5j + x - 8 in closed form."""
    rng = np.random.default_rng(seed)
    w = rng.uniform(-1.0, 1.0, (E, 32 * NT, 32 * KT))
    for x in range(E):
        for i in range(NT):
            for j in range(KT):
                t = w[x, 32 * i:32 * i + 32, 32 * j:32 * j + 32]
                t[(7 * i + j) % 32, (5 * j + i) % 32] = 1.0
                t *= 2.0 ** (3 * i - 5 * j + x)
    return w


def test_mx_weight_32x32_dequantise_tile_by_tile():
    """Quantise then dequantise tiles whose scales differ by powers of two:
    the exponents take their closed form, the dequantised tensor equals a
    loop over tiles that multiplies each tile's codes by its own 2^e, and
    every element that did not saturate is within half an E4M3 step (in its
    own binade) of the input.  A broadcast over the wrong axis, or the N and
    K tile axes exchanged (3 x 5 tiles), changes scales by powers of two and
    fails the loop and the half-step bound."""
    E, NT, KT = 2, 3, 5
    w = _tile_scaled_weight(E, NT, KT)
    q, e = fm.mx_quantize_weight_32x32(w)
    assert e.shape == (E, NT, KT)
    for x in range(E):
        for i in range(NT):
            for j in range(KT):
                assert e[x, i, j] == 3 * i - 5 * j + x - 8
    deq = fm.mx_dequantize_weight_32x32(q, e)
    loop = np.empty_like(w)
    for x in range(E):
        for i in range(NT):
            for j in range(KT):
                sl = (x, slice(32 * i, 32 * i + 32), slice(32 * j, 32 * j + 32))
                loop[sl] = q[sl] * 2.0 ** int(e[x, i, j])
    np.testing.assert_array_equal(deq, loop)
    # half an E4M3 step of the scaled value, in its own binade (subnormal
    # quantum 2^-9 below 2^-6), times the tile scale
    s = np.repeat(np.repeat(np.ldexp(1.0, e), 32, axis=1), 32, axis=2)
    y = np.abs(w) / s
    binade = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half_step = np.ldexp(1.0, (binade - 4).astype(int)) * s
    ok = y <= 448.0
    assert ok.mean() > 0.8
    assert np.all(np.abs(deq - w)[ok] <= half_step[ok])
    # saturated elements keep their sign at the largest code
    assert np.all(np.abs(deq[~ok]) == 448.0 * s[~ok])



# -------------------------------------------------------------------- SiLU

def test_silu_closed_form(golden_dir):
    g = _load(golden_dir, "silu_closed_form.json")
    for z, v in g["silu"]:
        assert moe.silu(z) == pytest.approx(v, rel=1e-15, abs=1e-300)
    for z, v in g["silu_grad"]:
        assert moe.silu_grad(z) == pytest.approx(v, rel=1e-14)


def test_silu_grad_is_derivative():
    z = np.linspace(-8, 8, 161)
    h = 1e-6
    fd = (moe.silu(z + h) - moe.silu(z - h)) / (2 * h)
    np.testing.assert_allclose(moe.silu_grad(z), fd, rtol=1e-8, atol=1e-9)


# ------------------------------------------------------------------ routing

def test_offsets_worked_example(golden_dir):
    g = _load(golden_dir, "offsets_worked_example.json")
    counts = g["counts"]
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)])
    ids = np.random.default_rng(5).permutation(ids).reshape(-1, 1)
    rt = moe.route(ids, len(counts), pad=1)
    assert rt.counts.tolist() == counts
    assert rt.offsets.tolist() == g["offsets"]
    for e, (a, b) in enumerate(g["expert_row_ranges"]):
        assert np.all(ids.reshape(-1)[rt.perm[a:b]] == e)


@pytest.mark.parametrize("T,K,E,pad", [(1, 1, 1, 32), (37, 3, 5, 32), (200, 6, 64, 32), (50, 2, 8, 1)])
def test_route_matches_stable_argsort(T, K, E, pad):
    rng = np.random.default_rng(T * 7 + E)
    ids = rng.integers(-1, E, size=(T, K))
    ids[0, 0] = E + 3          # out of range -> inactive + flagged
    if T > 1:
        ids[1, :] = -1         # an all-inactive token
    rt = moe.route(ids, E, pad)
    flat = ids.reshape(-1)
    active = (flat >= 0) & (flat < E)
    assert rt.counts.sum() == active.sum() == rt.num_active
    assert rt.bad_ids.tolist() == ((flat < -1) | (flat >= E)).tolist()
    # expected order: stable argsort of the IDs over the active routes
    act_idx = np.nonzero(active)[0]
    order = act_idx[np.argsort(flat[act_idx], kind="stable")]
    got = rt.perm[rt.perm >= 0]
    np.testing.assert_array_equal(got, order)
    assert np.all(np.diff(rt.poffsets) % pad == 0)
    assert np.all(np.diff(rt.poffsets) - rt.counts < pad)
    for e in range(E):
        a = rt.poffsets[e]
        seg = rt.perm[a:rt.poffsets[e + 1]]
        assert np.all(seg[:rt.counts[e]] >= 0) and np.all(seg[rt.counts[e]:] == -1)
    # inverse permutation
    assert np.all(rt.inv[~active] == -1)
    np.testing.assert_array_equal(rt.perm[rt.inv[active]], act_idx)


# ------------------------------------------------------------------ forward

def _case(T, D, F, E, K, seed, inactive=0.1):
    rng = np.random.default_rng(seed)
    x = fm.round_bf16(rng.standard_normal((T, D)))
    w13 = fm.round_bf16(rng.standard_normal((E, 2 * F, D)) / np.sqrt(D))
    w2 = fm.round_bf16(rng.standard_normal((E, D, F)) / np.sqrt(F))
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int64)
    s = rng.uniform(0.05, 1.0, (T, K)).astype(np.float32)
    off = rng.uniform(size=(T, K)) < inactive
    ids[off] = -1
    s[off] = 0.0
    return x, ids, s, w13, w2


@pytest.mark.parametrize("precision", ["f64", "bf16", "mxfp8"])
def test_routed_forward_matches_per_token_loop(precision):
    x, ids, s, w13, w2 = _case(40, 64, 96, 6, 3, 11)
    ids[7, :] = -1
    init = fm.round_bf16(np.random.default_rng(12).standard_normal(x.shape))
    st = moe.forward(x, ids, s, w13, w2, precision, out_init=init)
    ref = moe.forward_per_token(x, ids, s, w13, w2, precision, out_init=init)
    ref = np.stack([ref[t] for t in range(x.shape[0])])
    tol = 1e-12 if precision == "f64" else 1e-2
    err = np.max(np.abs(st["out"] - ref)) / np.max(np.abs(ref))
    assert err <= tol
    if precision != "f64":
        # rounding points make most outputs identical, not just close
        assert np.mean(st["out"] == ref) > 0.97


def test_single_expert_is_dense_swiglu():
    """E=1, K=1, score=1 reduces to the dense SwiGLU FFN W2 (SiLU(Wg x) * (Wu x))."""
    x, _, _, w13, w2 = _case(9, 32, 48, 1, 1, 13)
    ids = np.zeros((9, 1), np.int64)
    for score in (1.0, 0.5):
        s = np.full((9, 1), score, np.float32)
        out = moe.forward(x, ids, s, w13, w2, "f64")["out"]
        wg, wu = w13[0][:48], w13[0][48:]
        g = x @ wg.T
        u = x @ wu.T
        h = g / (1 + np.exp(-g)) * u
        np.testing.assert_allclose(out, score * (h @ w2[0].T), rtol=1e-12, atol=1e-14)


def test_inactive_routes_contribute_nothing():
    x, ids, s, w13, w2 = _case(16, 32, 32, 4, 2, 14, inactive=0.0)
    ids[3, :] = -1
    s[3, :] = 0.0
    for p in ("f64", "bf16", "mxfp8"):
        st = moe.forward(x, ids, s, w13, w2, p)
        assert np.all(st["out"][3] == 0.0)
    # a -1 route is ignored whatever score it carries
    ids2, s2 = ids.copy(), s.copy()
    ids2[5, 1] = -1
    s2[5, 1] = 0.7
    s3 = s2.copy()
    s3[5, 1] = 0.0
    a = moe.forward(x, ids2, s2, w13, w2, "bf16")["out"]
    b = moe.forward(x, ids2, s3, w13, w2, "bf16")["out"]
    np.testing.assert_array_equal(a, b)


def test_expert_relabelling_is_equivariant():
    x, ids, s, w13, w2 = _case(24, 32, 32, 5, 2, 15)
    p = np.array([3, 0, 4, 1, 2])           # new label of old expert e is p[e]
    ids2 = np.where(ids >= 0, p[np.maximum(ids, 0)], -1)
    w13b = np.empty_like(w13)
    w2b = np.empty_like(w2)
    w13b[p], w2b[p] = w13, w2
    for prec in ("bf16", "mxfp8"):
        a = moe.forward(x, ids, s, w13, w2, prec)["out"]
        b = moe.forward(x, ids2, s, w13b, w2b, prec)["out"]
        np.testing.assert_array_equal(a, b)


# ----------------------------------------------------------------- backward

def test_backward_matches_finite_differences():
    T, D, F, E, K = 6, 5, 4, 3, 2
    x, ids, s, w13, w2 = _case(T, D, F, E, K, 16, inactive=0.0)
    ids[2, 1] = -1
    s[2, 1] = 0.0
    rng = np.random.default_rng(17)
    dY = rng.standard_normal((T, D))

    def loss(x_, w13_, w2_):
        return float(np.sum(dY * moe.forward(x_, ids, s, w13_, w2_, "f64")["out"]))

    st = moe.forward(x, ids, s, w13, w2, "f64")
    g = moe.backward(st, dY, w13, w2)
    h = 1e-6

    def fd(arr, idx, which):
        a1, a2 = arr.copy(), arr.copy()
        a1[idx] += h
        a2[idx] -= h
        args1 = {"x": (a1, w13, w2), "w13": (x, a1, w2), "w2": (x, w13, a1)}[which]
        args2 = {"x": (a2, w13, w2), "w13": (x, a2, w2), "w2": (x, w13, a2)}[which]
        return (loss(*args1) - loss(*args2)) / (2 * h)

    for idx in np.ndindex(x.shape):
        assert g["dX"][idx] == pytest.approx(fd(x, idx, "x"), rel=1e-6, abs=1e-8)
    for idx in list(np.ndindex(w13.shape))[::3]:
        assert g["dW13"][idx] == pytest.approx(fd(w13, idx, "w13"), rel=1e-6, abs=1e-8)
    for idx in list(np.ndindex(w2.shape))[::2]:
        assert g["dW2"][idx] == pytest.approx(fd(w2, idx, "w2"), rel=1e-6, abs=1e-8)
    # score gradient: d loss / d s(t,k); inactive routes get none
    for t, k in np.ndindex(s.shape):
        s1, s2 = s.astype(np.float64).copy(), s.astype(np.float64).copy()
        s1[t, k] += h
        s2[t, k] -= h
        f1 = float(np.sum(dY * moe.forward(x, ids, s1, w13, w2, "f64")["out"]))
        f2 = float(np.sum(dY * moe.forward(x, ids, s2, w13, w2, "f64")["out"]))
        assert g["dp"][t, k] == pytest.approx((f1 - f2) / (2 * h), rel=1e-6, abs=1e-8)
    assert g["dp"][2, 1] == 0.0


def test_backward_inactive_routes_get_no_gradient():
    x, ids, s, w13, w2 = _case(20, 32, 32, 5, 2, 18, inactive=0.0)
    ids[ids == 4] = 0            # expert 4 is reached by no active route...
    ids[9, :] = [4, -1]          # ...except one that we then disable
    ids[9, 0] = -1
    s[9, :] = 0.0
    dY = np.random.default_rng(19).standard_normal(x.shape)
    for p in ("f64", "bf16", "mxfp8"):
        st = moe.forward(x, ids, s, w13, w2, p)
        g = moe.backward(st, dY, w13, w2)
        assert np.all(g["dX"][9] == 0.0)
        assert np.all(g["dW13"][4] == 0.0) and np.all(g["dW2"][4] == 0.0)


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_rounded_backward_tracks_exact_backward(precision):
    x, ids, s, w13, w2 = _case(64, 64, 64, 4, 2, 20)
    dY = fm.round_bf16(np.random.default_rng(21).standard_normal(x.shape))
    ex = moe.backward(moe.forward(x, ids, s, w13, w2, "f64"), dY, w13, w2)
    rd = moe.backward(moe.forward(x, ids, s, w13, w2, precision), dY, w13, w2)
    # MXFP8: the OCP scale rule puts a block's maximum in [256, 512) after
    # scaling, so a maximum scaled past 448 is clipped by up to 12.5%; a
    # weight gradient dominated by one row inherits that clipping.
    tol = 0.02 if precision == "bf16" else 0.15
    for k in ("dX", "dW13", "dW2"):
        err = np.max(np.abs(rd[k] - ex[k])) / np.max(np.abs(ex[k]))
        assert err < tol, (k, err)


# ------------------------------------------------------ clamped SwiGLU, 1x32 weights
# "Meta Dist-MoE: Open-Source Fused MoE Kernels for Blackwell", "Supported
# modes": plain and clamped SwiGLU; 1x32 weight blocks for inference.

def test_clamped_swiglu_closed_form():
    # SiLU(1) = 1 / (1 + e^-1) = 0.7310585786300049; SiLU(-5) = -5 / (1 + e^5)
    g = np.array([2.0, -5.0, 0.5, 3.0])
    u = np.array([3.0, -10.0, 0.25, -0.5])
    h = moe.swiglu(g, u, limit=1.0)
    assert h[0] == pytest.approx(0.7310585786300049 * 1.0, rel=1e-15)      # g -> 1, u -> 1
    assert h[1] == pytest.approx((-5.0 / (1.0 + np.exp(5.0))) * -1.0, rel=1e-15)   # u -> -1
    assert h[2] == pytest.approx(0.5 / (1.0 + np.exp(-0.5)) * 0.25, rel=1e-15)    # inside: unchanged
    assert h[3] == pytest.approx(0.7310585786300049 * -0.5, rel=1e-15)     # only g clamped
    # limit 0 is the plain SwiGLU, and a limit above every value changes nothing
    assert np.array_equal(moe.swiglu(g, u, 0.0), moe.silu(g) * u)
    assert np.array_equal(moe.swiglu(g, u, 100.0), moe.silu(g) * u)


def test_clamped_swiglu_grad_matches_finite_differences():
    rng = np.random.default_rng(31)
    L = 0.8
    g = rng.uniform(-3, 3, 200)
    u = rng.uniform(-3, 3, 200)
    keep = (np.abs(g - L) > 1e-3) & (np.abs(np.abs(u) - L) > 1e-3)   # away from the kinks
    g, u = g[keep], u[keep]
    dh = rng.standard_normal(g.shape)
    dg, du = moe.swiglu_grad(g, u, dh, L)
    h = 1e-7
    fd_g = (moe.swiglu(g + h, u, L) - moe.swiglu(g - h, u, L)) / (2 * h) * dh
    fd_u = (moe.swiglu(g, u + h, L) - moe.swiglu(g, u - h, L)) / (2 * h) * dh
    assert np.allclose(dg, fd_g, rtol=1e-6, atol=1e-9)
    assert np.allclose(du, fd_u, rtol=1e-6, atol=1e-9)
    assert np.all(dg[g > L] == 0.0) and np.all(du[np.abs(u) > L] == 0.0)


def test_clamped_layer_backward_matches_finite_differences():
    T, D, F, E, K = 6, 5, 4, 3, 2
    x, ids, s, w13, w2 = _case(T, D, F, E, K, 16, inactive=0.0)
    x = x * 3.0                   # large enough that some gate / up values clip
    L = 0.3
    dY = np.random.default_rng(33).standard_normal((T, D))
    st = moe.forward(x, ids, s, w13, w2, "f64", swiglu_limit=L)
    F_ = st["F"]
    g1, u1 = st["h1"][:, :F_], st["h1"][:, F_:]
    assert st["clip"][0] > 0 and st["clip"][1] > 0
    assert np.min(np.abs(g1 - L)) > 1e-5 and np.min(np.abs(np.abs(u1) - L)) > 1e-5
    grads = moe.backward(st, dY, w13, w2)
    h = 1e-7

    def loss(x_):
        return float(np.sum(dY * moe.forward(x_, ids, s, w13, w2, "f64", swiglu_limit=L)["out"]))

    for idx in np.ndindex(x.shape):
        a1, a2 = x.copy(), x.copy()
        a1[idx] += h
        a2[idx] -= h
        assert grads["dX"][idx] == pytest.approx((loss(a1) - loss(a2)) / (2 * h), rel=1e-5, abs=1e-8)


def test_clip_counts_count_the_clamped_values():
    h1 = np.array([[0.5, 2.0, -3.0, 0.1], [1.5, -1.0, 0.2, -1.5]])   # F = 2: gate cols 0-1, up cols 2-3
    assert moe.clip_counts(h1, 2, 1.0) == (2, 2)    # gate > 1: 2.0, 1.5; |up| > 1: -3.0, -1.5
    assert moe.clip_counts(h1, 2, 0.0) == (0, 0)


def test_weight_1x32_blocks_are_per_row():
    rng = np.random.default_rng(35)
    w = rng.standard_normal((64, 128))
    q = moe.prepare_weight(w, "mxfp8", "1x32")
    w2 = w.copy()
    w2[5, 40] = 1e4               # an outlier in row 5, block 1
    q2 = moe.prepare_weight(w2, "mxfp8", "1x32")
    changed = np.argwhere(q2 != q)
    # only that row's 32-value block is affected (1x32), not its 32x32 tile
    assert set(map(tuple, changed[:, :1].tolist())) == {(5,)}
    assert changed[:, 1].min() >= 32 and changed[:, 1].max() < 64
    t1, t2 = moe.prepare_weight(w, "mxfp8"), moe.prepare_weight(w2, "mxfp8")
    assert len(set(np.argwhere(t2 != t1)[:, 0].tolist())) > 1     # 32x32: the whole tile moves
    # every 1x32 block of every row is the MX quantisation of that block alone
    for r in (0, 5, 63):
        for b in range(4):
            blk = w[r, 32 * b:32 * (b + 1)][None, :]
            assert np.array_equal(q[r, 32 * b:32 * (b + 1)], fm.mx_fake_quant(blk, axis=-1)[0])


# ---------------------------------------------------------- post-expert RMSNorm

def test_post_norm_constant_row_closed_form():
    """A row of equal values a: mean(x^2) = a^2, so y = gamma * a / sqrt(a^2 + eps)
    whatever D is."""
    from oracle import post_norm as pn
    rng = np.random.default_rng(5)
    for D in (8, 96):
        gamma = rng.normal(size=D)
        for a, eps in ((0.75, 1e-6), (-3.0, 0.5), (2.0 ** -10, 1e-3)):
            y, r = pn.forward(np.full((1, D), a), gamma, eps, rounding=False)
            np.testing.assert_allclose(y[0], gamma * a / math.sqrt(a * a + eps), rtol=1e-14, atol=0)
            assert r[0] == pytest.approx(1.0 / math.sqrt(a * a + eps), rel=1e-14)


def test_post_norm_zero_row():
    """An all-zero row (every route inactive, no shared expert) stays zero, and
    its gradient is gamma * dy / sqrt(eps) (c = 0)."""
    from oracle import post_norm as pn
    D, eps = 16, 1e-5
    gamma = np.linspace(-1.0, 1.5, D)
    dy = np.linspace(0.3, -0.7, D)[None, :]
    y, _ = pn.forward(np.zeros((1, D)), gamma, eps, rounding=False)
    assert np.all(y == 0.0)
    dx, dg = pn.backward(np.zeros((1, D)), gamma, eps, dy, rounding=False)
    np.testing.assert_allclose(dx[0], gamma * dy[0] / math.sqrt(eps), rtol=1e-14)
    assert np.all(dg == 0.0)


def test_post_norm_scale_invariant_without_eps():
    """With eps = 0 the map forgets the row's scale: y(alpha x) = y(x)."""
    from oracle import post_norm as pn
    rng = np.random.default_rng(6)
    x = rng.normal(size=(3, 24))
    gamma = rng.normal(size=24)
    y1, _ = pn.forward(x, gamma, 0.0, rounding=False)
    for alpha in (1e-3, 7.0, 2.0 ** 20):
        y2, _ = pn.forward(alpha * x, gamma, 0.0, rounding=False)
        np.testing.assert_allclose(y2, y1, rtol=1e-12)


def test_post_norm_backward_matches_finite_differences():
    """dx and dgamma against central differences of L = sum(dy * y) in fp64."""
    from oracle import post_norm as pn
    rng = np.random.default_rng(7)
    T, D, eps = 3, 8, 1e-3
    x = rng.normal(size=(T, D))
    gamma = rng.normal(size=D)
    dy = rng.normal(size=(T, D))
    dx, dg = pn.backward(x, gamma, eps, dy, rounding=False)

    def loss(xv, gv):
        return float(np.sum(dy * pn.forward(xv, gv, eps, rounding=False)[0]))

    h = 1e-6
    num_dx = np.zeros_like(x)
    for t in range(T):
        for d in range(D):
            e = np.zeros_like(x)
            e[t, d] = h
            num_dx[t, d] = (loss(x + e, gamma) - loss(x - e, gamma)) / (2 * h)
    num_dg = np.zeros(D)
    for d in range(D):
        e = np.zeros(D)
        e[d] = h
        num_dg[d] = (loss(x, gamma + e) - loss(x, gamma - e)) / (2 * h)
    np.testing.assert_allclose(dx, num_dx, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dg, num_dg, rtol=1e-6, atol=1e-8)


def test_post_norm_rounds_outputs_to_bf16():
    from oracle import post_norm as pn
    rng = np.random.default_rng(8)
    x = fm.round_bf16(rng.normal(size=(4, 32)))
    gamma = fm.round_bf16(rng.normal(size=32))
    y, _ = pn.forward(x, gamma, 1e-6)
    np.testing.assert_array_equal(y, fm.round_bf16(y))
    yx, _ = pn.forward(x, gamma, 1e-6, rounding=False)
    assert np.max(np.abs(y - yx) / np.maximum(np.abs(yx), 1e-30)) <= 2.0 ** -8


# ------------------------------------------------------------ bounded samples

@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_sample_reproduces_the_full_problem_for_its_experts(precision):
    """oracle/sample.py, against the full oracle by brute force: with the
    routes restricted to chosen experts, each chosen expert keeps its rows,
    its h1 and its weight gradients exactly, and a token whose active routes
    all reach chosen experts keeps its out, dX and score gradients."""
    from oracle import sample as osample
    T, D, F, E, K = 96, 128, 128, 8, 2
    x, ids, s, w13, w2 = _case(T, D, F, E, K, 41)
    dY = fm.round_bf16(np.random.default_rng(42).standard_normal((T, D)))
    full = moe.forward(x, ids, s, w13, w2, precision)
    fg = moe.backward(full, dY, w13, w2)
    experts = [5, 1, 6]
    res = osample.run(x, ids, s, w13[experts], w2[experts], experts, precision, dY=dY)
    st, g = res["state"], res["grads"]
    assert np.array_equal(res["ids"] >= 0, np.isin(ids, experts))
    for i, e in enumerate(experts):
        a, b = full["routing"].poffsets[e], full["routing"].poffsets[e + 1]
        c, d = st["routing"].poffsets[i], st["routing"].poffsets[i + 1]
        assert b - a == d - c
        np.testing.assert_array_equal(st["h1"][c:d], full["h1"][a:b])
        np.testing.assert_array_equal(g["dW13"][i], fg["dW13"][e])
        np.testing.assert_array_equal(g["dW2"][i], fg["dW2"][e])
    whole = np.all((ids < 0) | np.isin(ids, experts), axis=1) & np.any(np.isin(ids, experts), axis=1)
    assert whole.sum() >= 5
    np.testing.assert_array_equal(st["out"][whole], full["out"][whole])
    np.testing.assert_array_equal(g["dX"][whole], fg["dX"][whole])
    np.testing.assert_array_equal(g["dp"][whole], fg["dp"][whole])
    assert osample.useful_flops(res["ids"], D, F, True) == 18.0 * np.isin(ids, experts).sum() * D * F


@pytest.mark.parametrize("case", ["all_to_one", "all_inactive"])
def test_route_degenerate_distributions(case):
    """The routing matrix's degenerate corners: every route to one expert of
    eight (the others empty), and no active route at all."""
    T, K, E = 300, 2, 8
    ids = np.full((T, K), 5 if case == "all_to_one" else -1, dtype=np.int64)
    rt = moe.route(ids, E)
    n = T * K if case == "all_to_one" else 0
    assert rt.num_active == n and rt.counts.tolist() == [n if e == 5 else 0 for e in range(E)]
    pad = -(-n // 32) * 32
    assert rt.poffsets.tolist() == [0] * 6 + [pad] * 3
    np.testing.assert_array_equal(rt.perm[:n], np.arange(n))          # flat order kept
    assert np.all(rt.perm[n:pad] == -1)
    np.testing.assert_array_equal(rt.inv, np.arange(T * K) if n else np.full(T * K, -1))
    x, _, s, w13, w2 = _case(T, 32, 32, E, K, 43, inactive=0.0)
    out = moe.forward(x, ids, s, w13, w2, "f64")["out"]
    if case == "all_inactive":
        assert np.all(out == 0.0)
    else:
        ref = moe.forward_per_token(x, ids, s, w13, w2, "f64")
        np.testing.assert_allclose(out, np.stack([ref[t] for t in range(T)]), rtol=1e-12, atol=1e-12)
