"""fp64 oracle of the post-expert RMSNorm.  TEST INFRASTRUCTURE ONLY (see
``oracle/__init__``).

"Meta Dist-MoE: Open-Source Fused MoE Kernels for Blackwell", "Supported
modes", lists a fused post-expert RMSNorm among the layer's features without
defining it.  Reading (also in the design notes): the layer's output row
x[t] -- the BF16 result of the score-weighted combine, after the shared
expert's output is added -- is normalised over the model width D with a
learned per-feature weight gamma, in the same pass:

    r[t]      = 1 / sqrt( mean_d x[t,d]^2 + eps )
    y[t,d]    = R( gamma[d] * x[t,d] * r[t] )

Backward, from dy = dL/dy (the chain rule through the three lines above,
written out; dr/dx_j = -r^3 x_j / D):

    g[t,d]    = gamma[d] * dy[t,d],   c[t] = mean_d g[t,d] x[t,d]
    dx[t,d]   = R( r[t] g[t,d] - x[t,d] r[t]^3 c[t] )
    dgamma[d] = sum_t dy[t,d] x[t,d] r[t]

R is BF16 rounding, or the identity when ``rounding`` is False (the
finite-difference pin uses that).  dgamma is left unrounded (it is an FP32
output).
"""

import numpy as np

from . import formats as fm


def _r(v, rounding):
    return fm.round_bf16(v) if rounding else v


def rstd(x, eps):
    """r[t] = 1 / sqrt(mean_d x[t,d]^2 + eps)."""
    x = np.asarray(x, np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)


def forward(x, gamma, eps, rounding=True):
    """y = R(gamma * x * r); returns (y, r)."""
    x = np.asarray(x, np.float64)
    gamma = np.asarray(gamma, np.float64)
    r = rstd(x, eps)
    return _r(gamma[None, :] * x * r[:, None], rounding), r


def backward(x, gamma, eps, dy, rounding=True):
    """dx = R(r g - x r^3 c) with g = gamma dy, c = mean_d(g x);
    dgamma = sum_t dy x r.  Returns (dx, dgamma)."""
    x = np.asarray(x, np.float64)
    gamma = np.asarray(gamma, np.float64)
    dy = np.asarray(dy, np.float64)
    r = rstd(x, eps)
    g = gamma[None, :] * dy
    c = np.mean(g * x, axis=-1)
    dx = r[:, None] * g - x * (r ** 3 * c)[:, None]
    dgamma = np.sum(dy * x * r[:, None], axis=0)
    return _r(dx, rounding), dgamma
