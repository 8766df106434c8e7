"""Number formats of the MoE path, written from their definitions (fp64).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources
-------
* Dist-MoE visual explainer, section 02 "Expert Computation and Tensor
  Precision": E4M3 has 4 exponent and 3 fraction bits with largest finite
  magnitude 448; E8M0 is a one-byte power-of-two scale; MXFP8 keeps one E8M0
  scale per 32 logical values, and the producer picks the scale.
* Same section, "Quantization Axes for Forward and Backward": activations are
  scaled along the contraction axis (1x32 row bundles for FPROP/DGRAD, 32x1
  column bundles for WGRAD); static weights use 32x32 blocks whose one scale
  serves both orientations.

Readings where the pages leave a step open
------------------------------------------
* Scale rule (the pages give none): the OCP MX v1.0 rule that the name MXFP8
  refers to -- shared exponent = floor(log2(amax)) - 8 (8 = largest E4M3
  exponent), clamped to the E8M0 range [-127, 127]; amax = 0 gives -127.
  Elements are v * 2^-e rounded to nearest-even in E4M3 and saturated to
  +-448.
* E4M3 is the "FN" variant: bias 7, no infinities, S.1111.111 is NaN, the
  smallest subnormal is 2^-9.
* E8M0: bias 127, 0xFF is NaN (never produced here).
"""

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8          # largest unbiased exponent of a finite E4M3 value
MX_BLOCK = 32


def round_to_binary(x, frac_bits, emin, max_finite=None, saturate=False):
    """Round float64 ``x`` to nearest-even in a binary format.

    The format has ``frac_bits`` stored fraction bits, smallest normal
    exponent ``emin`` and gradual underflow (subnormals spaced
    2^(emin - frac_bits)).  Values above ``max_finite`` saturate to it when
    ``saturate`` else become +-inf.  The division by the quantum is exact
    (power of two) and ``np.round`` rounds halves to even.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(np.abs(x))           # |x| = m 2^e, m in [0.5, 1)
    e = np.maximum(e - 1, emin)          # floor(log2|x|), floored at emin
    quantum = np.ldexp(1.0, e - frac_bits)
    r = np.round(x / quantum) * quantum
    if max_finite is not None:
        over = np.abs(r) > max_finite
        if saturate:
            r = np.where(over, np.copysign(max_finite, x), r)
        else:
            r = np.where(over, np.copysign(np.inf, x), r)
    return r


# ----------------------------------------------------------------- BF16 / FP32

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(x):
    """Round to BF16 (8 exponent bits, 7 fraction bits), nearest-even."""
    return round_to_binary(x, 7, -126, BF16_MAX, saturate=False)


def round_fp32(x):
    """Round to IEEE binary32, nearest-even."""
    return round_to_binary(x, 23, -126, np.finfo(np.float32).max, saturate=False)


def bf16_bits_to_f64(bits):
    """Decode BF16 bit patterns (uint16) to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Encode float64 values that are already BF16-representable as uint16."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------- E4M3

def round_e4m3(x):
    """Nearest-even E4M3FN value of ``x``, saturating to +-448."""
    return round_to_binary(x, 3, -6, E4M3_MAX, saturate=True)


def e4m3_decode(codes):
    """Value of each E4M3FN byte (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = sign * np.ldexp(1.0 + man / 8.0, exp - 7)
    sub = sign * np.ldexp(man / 8.0, -6)
    v = np.where(exp == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e4m3_encode(values):
    """Byte of each E4M3FN-representable value (input must be on the grid)."""
    v = np.asarray(values, dtype=np.float64)
    sign = np.where(np.signbit(v), 0x80, 0).astype(np.int64)
    a = np.abs(v)
    _, e = np.frexp(a)
    e = e - 1                                   # floor(log2 a)
    is_sub = (a < 2.0 ** -6)
    exp_field = np.where(is_sub, 0, e + 7)
    man = np.where(is_sub, a / 2.0 ** -9, (a / np.ldexp(1.0, e) - 1.0) * 8.0)
    man = np.where(a == 0, 0, man)
    exp_field = np.where(a == 0, 0, exp_field)
    code = sign | (exp_field.astype(np.int64) << 3) | np.rint(man).astype(np.int64)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------- E8M0

def e8m0_decode(byte):
    """2^(b - 127) for each E8M0 byte (NaN for 0xFF)."""
    b = np.asarray(byte, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


def mx_shared_exponent(amax):
    """OCP MX shared exponent: floor(log2 amax) - 8, clamped to [-127, 127].

    amax = 0 gives -127 (E8M0 byte 0x00)."""
    a = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(a)
    e = (e - 1) - E4M3_EMAX
    e = np.where(a == 0, -127, e)
    return np.clip(e, -127, 127).astype(np.int64)


# ------------------------------------------------------------- MX quantisers

def mx_quantize(v, axis=-1):
    """MXFP8 quantisation of ``v`` in blocks of 32 consecutive values along
    ``axis`` (the contraction axis of the GEMM that consumes it).

    Returns ``(q, e)``: ``q`` holds the E4M3 element values (same shape as
    ``v``), ``e`` the shared exponents with the blocked axis shortened 32x.
    The dequantised tensor is ``q * 2^e`` broadcast over each block.
    """
    v = np.moveaxis(np.asarray(v, dtype=np.float64), axis, -1)
    n = v.shape[-1]
    assert n % MX_BLOCK == 0, "MX axis must be a multiple of 32"
    blk = v.reshape(v.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    amax = np.max(np.abs(blk), axis=-1)
    e = mx_shared_exponent(amax)
    q = round_e4m3(blk * np.ldexp(1.0, -e)[..., None])
    q = q.reshape(v.shape)
    return np.moveaxis(q, -1, axis), np.moveaxis(e, -1, axis)


def mx_dequantize(q, e, axis=-1):
    """q * 2^e with each exponent broadcast over its block of 32 along axis."""
    q = np.moveaxis(np.asarray(q, dtype=np.float64), axis, -1)
    e = np.moveaxis(np.asarray(e), axis, -1)
    scale = np.repeat(np.ldexp(1.0, e), MX_BLOCK, axis=-1)
    return np.moveaxis(q * scale, -1, axis)


def mx_fake_quant(v, axis=-1):
    """Dequantised MXFP8 copy of ``v`` (quantise along ``axis``, then expand)."""
    q, e = mx_quantize(v, axis)
    return mx_dequantize(q, e, axis)


def mx_quantize_weight_32x32(w):
    """Static-weight MXFP8 with one scale per 32x32 tile of the last two axes.

    Returns ``(q, e)`` with ``e`` of shape [..., N/32, K/32].  The same
    exponent serves the forward (1x32 along K) and the input-gradient
    (1x32 along N) orientation, so both share ``q``."""
    w = np.asarray(w, dtype=np.float64)
    *lead, n, k = w.shape
    assert n % MX_BLOCK == 0 and k % MX_BLOCK == 0
    t = w.reshape(tuple(lead) + (n // 32, 32, k // 32, 32))
    amax = np.max(np.abs(t), axis=(-3, -1))
    e = mx_shared_exponent(amax)
    q = round_e4m3(t * np.ldexp(1.0, -e)[..., :, None, :, None])
    return q.reshape(w.shape), e


def mx_dequantize_weight_32x32(q, e):
    *lead, n, k = q.shape
    s = np.ldexp(1.0, e)[..., :, None, :, None]
    return (q.reshape(tuple(lead) + (n // 32, 32, k // 32, 32)) * s).reshape(q.shape)


# ---------------------------------------------------------------- E2M1, NVFP4
#
# Dist-MoE explainer, section 02, "Expert Computation and Tensor Precision":
# E2M1 holds a sign, two exponent bits and one fraction bit in four bits;
# NVFP4 packs two E2M1 values per byte and uses E4M3 block scales plus
# global scales; NVFP4 inference quantises on the source side and publishes
# packed data, block scales and the row's inverse global scale.
#
# Readings where the pages leave a step open (the NVFP4 format's own
# conventions):
# * E2M1: exponent bias 1, no infinities or NaN; magnitudes 0, 0.5, 1, 1.5,
#   2, 3, 4, 6; round to nearest even, saturating to +-6.
# * Blocks of 16 consecutive values along the contraction axis, one E4M3
#   block scale each (a positive value, rounded to nearest even, saturating
#   to 448), and one FP32 global scale per row: g = amax(row) / (6 * 448), so
#   the largest block scale lands at 448 and the largest value at 6.
# * Every step is one FP32 operation, rounded to nearest even, in this order
#   (both sides of a parity test decide the codes with the same FP32 values):
#     g   = fp32(a_row / 2688)
#     s6g = fp32(6 * g)
#     sb  = E4M3(fp32(a_block / s6g))
#     d   = fp32(sb * g)
#     q   = E2M1(fp32(v / d))          (q = 0 where d = 0)
#   and v is represented by q * sb * g.  A zero row has g = 0 and all codes 0.

E2M1_MAX = 6.0
NVFP4_BLOCK = 16
NVFP4_GLOBAL_DIV = 6.0 * E4M3_MAX     # 2688: the largest E2M1 times the largest E4M3


def round_e2m1(x):
    """Nearest-even E2M1 value of ``x``, saturating to +-6."""
    return round_to_binary(x, 1, 0, E2M1_MAX, saturate=True)


def e2m1_decode(codes):
    """Value of each 4-bit E2M1 code (bit 3 sign, bits 2-1 exponent, bit 0
    fraction; exponent 0 is subnormal: 0 or 0.5)."""
    c = np.asarray(codes, dtype=np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    exp = (c >> 1) & 0x3
    man = c & 0x1
    return sign * np.where(exp == 0, man * 0.5, np.ldexp(1.0 + man / 2.0, exp - 1))


def e2m1_encode(values):
    """4-bit code of each E2M1-representable value (input on the grid)."""
    v = np.asarray(values, dtype=np.float64)
    sign = np.where(np.signbit(v), 0x8, 0)
    a = np.abs(v)
    _, e = np.frexp(a)
    e = e - 1                                   # floor(log2 a) for a > 0
    sub = a < 1.0
    exp_field = np.where(sub, 0, e + 1)
    man = np.where(sub, a / 0.5, (a / np.ldexp(1.0, e) - 1.0) * 2.0)
    code = sign | (exp_field.astype(np.int64) << 1) | np.rint(man).astype(np.int64)
    return np.where(a == 0, sign, code).astype(np.uint8)


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def nvfp4_quantize(v, axis=-1):
    """NVFP4 quantisation of ``v`` (values exactly representable in FP32)
    in blocks of 16 along ``axis``, with one global scale per row (all other
    axes).  Returns ``(q, sb, g)``: E2M1 values (shape of v), E4M3 block
    scales (the blocked axis shortened 16x) and FP32 row scales (the blocked
    axis removed), all as float64."""
    v = np.moveaxis(np.asarray(v, dtype=np.float64), axis, -1)
    n = v.shape[-1]
    assert n % NVFP4_BLOCK == 0, "NVFP4 axis must be a multiple of 16"
    v32 = _f32(v)
    assert np.array_equal(v32.astype(np.float64), v), "inputs must be FP32 values"
    a_row = np.max(np.abs(v32), axis=-1)
    g = _f32(a_row / np.float32(NVFP4_GLOBAL_DIV))
    s6g = _f32(np.float32(6.0) * g)
    blk = v32.reshape(v32.shape[:-1] + (n // NVFP4_BLOCK, NVFP4_BLOCK))
    a_blk = np.max(np.abs(blk), axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(s6g[..., None] > 0, _f32(a_blk / s6g[..., None]), np.float32(0.0))
    sb = _f32(round_e4m3(ratio.astype(np.float64)))
    d = _f32(sb * g[..., None])
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(d[..., None] > 0, _f32(blk / d[..., None]), np.float32(0.0))
    q = round_e2m1(y.astype(np.float64)).reshape(v.shape)
    return (np.moveaxis(q, -1, axis), np.moveaxis(sb.astype(np.float64), -1, axis),
            g.astype(np.float64))


def nvfp4_dequantize(q, sb, g, axis=-1):
    """q * sb * g with each block scale broadcast over its 16 values and the
    row scale over the row."""
    q = np.moveaxis(np.asarray(q, dtype=np.float64), axis, -1)
    sb = np.moveaxis(np.asarray(sb, dtype=np.float64), axis, -1)
    return np.moveaxis(q * np.repeat(sb, NVFP4_BLOCK, axis=-1) * np.asarray(g)[..., None], -1, axis)


def nvfp4_fake_quant(v, axis=-1):
    """Dequantised NVFP4 copy of ``v`` (FP32 values) along ``axis``."""
    q, sb, g = nvfp4_quantize(v, axis)
    return nvfp4_dequantize(q, sb, g, axis)
