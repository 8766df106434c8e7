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
