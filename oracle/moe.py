"""fp64 oracle of the dropless routed-expert MoE layer (one GPU, all experts local).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What it computes
----------------
Forward, for every token t (blog "Mixture of Experts: How Routing Becomes GPU
Computation", section 2, "SwiGLU forward: compute and combine expert
outputs"; Dist-MoE explainer section 02, h1 = W13 x = [g; u],
h2 = SiLU(g) * u, h3 = W2 h2):

    out[t] = R( init[t] + sum_k [id(t,k) active] * s(t,k) * h3(t,k) )
    h3 = R( W2[e] . q2(h2) ),  h2 = SiLU(g) * u,  [g; u] = R( W13[e] . q1(x[t]) )

with e = id(t,k), R = BF16 rounding (identity in the "f64" mode), q1/q2 the
activation quantiser of the precision (identity, BF16 rounding, or MXFP8
along the contraction axis) and weights quantised once (MXFP8: 32x32 blocks).

Backward (blog section 2, "SwiGLU backward: the complete expert path" and
"Grouped GEMM backward: one projection"; Dist-MoE explainer section 05 for the
op order W2 DGRAD/WGRAD, SwiGLU backward, W13 DGRAD/WGRAD, K-reduction):

    dh3 = q(fp32(s * dY[t]))           (row bundle along D, column bundle along rows)
    dh2 = dh3_row . W2[e]              (kept unrounded: fused into the SwiGLU backward)
    dg  = dh2 * u * SiLU'(g),  du = dh2 * SiLU(g),  dh1 = [dg; du]
    dxr = R( q(dh1)_row . W13[e] ),   dX[t] = R( init[t] + sum_k dxr(t,k) )
    dW2[e]  = Rw( sum_rows dh3_colT . h2_col )
    dW13[e] = Rw( sum_rows dh1_colT . x_col )
    dp(t,k) = <h3(t,k), dY[t]>        (score gradient, unrounded)

Readings of the pages (each also listed in the design notes)
------------------------------------------------------------
* Routing order: stable by flattened route index t*K+k within an expert
  (the blog packs with a stable argsort over the flattened [T,K] IDs).
* ID -1 (or any ID outside [0,E)) is an inactive route: no row, no
  contribution, no gradient, whatever its score (Dist-MoE explainer section 01
  "Inputs, shapes, and inactive routes").
* Each expert's rows are padded to a multiple of 32 (the MX block along
  rows that the WGRAD column bundles need); pad rows are zero.
* h1 is rounded to BF16 before the SwiGLU; h2 is formed once (fp64 here) and
  quantised once; h3 is rounded to BF16; the score multiply and the K-sum
  are done wide and rounded once.
* dh3 is the fp32 product s*dY (the blog forms it with ``.float()``) and is
  then rounded/quantised, so the quantised codes are decided in the same
  precision as on the GPU.
* MXFP8 WGRAD operands are column bundles: the unquantised source quantised
  in 32-row blocks aligned to each expert's first row.
* Clamped SwiGLU ("Meta Dist-MoE: Open-Source Fused MoE Kernels for
  Blackwell", "Supported modes", lists plain and clamped SwiGLU without
  defining the clamp): with a limit L > 0, g is clamped from above and u on
  both sides before the plain SwiGLU, h2 = SiLU(min(g, L)) * clamp(u, -L, L),
  on the BF16-rounded h1; the backward passes a gradient where the input lies
  inside the clamp range, bounds included (the convention of a clamp's
  subgradient).  L = 0 is the plain SwiGLU.
* Inference weights with 1x32 blocks (same section: "32x32 blocks for MXFP8
  training-compatible values or 1x32 for inference"): one scale per 32
  consecutive values of a weight row along the contraction axis.
* NVFP4 (inference only; Dist-MoE explainer, section 08, "Public API and
  Supported Modes": NVFP4 inference with prepared weights): weights, x rows
  and h2 rows quantised along their contraction axis in blocks of 16 with
  E4M3 block scales and one FP32 global scale per row (``formats``); h1 and
  h3 are rounded to BF16 as in the other modes.
"""

from collections import namedtuple

import numpy as np

from . import formats as fm

PAD = 32

Routing = namedtuple(
    "Routing", "counts offsets poffsets perm inv bad_ids num_active")


# ------------------------------------------------------------------ SwiGLU

def silu(z):
    """SiLU(z) = z / (1 + e^-z)  (blog section 1; Dist-MoE explainer section 02)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def silu_grad(z):
    """d/dz SiLU(z) = s (1 + z (1 - s)), s = sigmoid(z) (blog section 2, silu_grad)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


# ------------------------------------------------------------------ routing

def route(ids, num_experts, pad=PAD):
    """Group the flattened routes by expert (blog section 2, "Packing").

    A counting sort: per-expert counts, exclusive prefix sums (``offsets``
    unpadded, ``poffsets`` with every expert padded to a multiple of ``pad``),
    then one pass over the routes in flat order placing route i = t*K+k at
    the next free row of its expert, which keeps the order stable.

    Returns ``Routing``: counts[E], offsets[E+1], poffsets[E+1],
    perm[poffsets[E]] (route index of each padded row, -1 for pad rows),
    inv[T*K] (row of each route, -1 if inactive), bad_ids (mask of IDs
    outside [-1, E)), num_active.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    E = int(num_experts)
    active = (flat >= 0) & (flat < E)
    bad = (flat < -1) | (flat >= E)
    counts = np.zeros(E, dtype=np.int64)
    for i in range(flat.size):
        if active[i]:
            counts[flat[i]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    poffsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
        poffsets[e + 1] = poffsets[e] + (counts[e] + pad - 1) // pad * pad
    perm = np.full(poffsets[E], -1, dtype=np.int64)
    inv = np.full(flat.size, -1, dtype=np.int64)
    nxt = poffsets[:E].copy()
    for i in range(flat.size):
        if active[i]:
            e = flat[i]
            perm[nxt[e]] = i
            inv[i] = nxt[e]
            nxt[e] += 1
    return Routing(counts, offsets, poffsets, perm, inv, bad, int(active.sum()))


# ------------------------------------------------------- precision helpers

PRECISIONS = ("f64", "bf16", "mxfp8", "nvfp4")


def _round_out(v, precision):
    """Rounding of a stored BF16 tensor (identity in the exact mode)."""
    return v if precision == "f64" else fm.round_bf16(v)


def _q_row(v, precision):
    """Activation quantiser along the last (feature) axis: FPROP/DGRAD operand.
    NVFP4 (inference): the value is first rounded to FP32, the precision in
    which the GPU holds it, then quantised by the FP32 steps of the format."""
    if precision == "f64":
        return v
    if precision == "bf16":
        return fm.round_bf16(v)
    if precision == "nvfp4":
        return fm.nvfp4_fake_quant(fm.round_fp32(v), axis=-1)
    return fm.mx_fake_quant(v, axis=-1)


def _q_col(v, precision):
    """Activation quantiser along rows (axis 0, 32-row blocks): WGRAD operand."""
    if precision == "f64":
        return v
    if precision == "bf16":
        return fm.round_bf16(v)
    return fm.mx_fake_quant(v, axis=0)


def prepare_weight(w_e, precision, blocks="32x32"):
    """One expert's weight [N, K] as the GEMMs consume it: MXFP8 with 32x32
    blocks (training) or 1x32 blocks along K (inference)."""
    w_e = np.asarray(w_e, dtype=np.float64)
    if precision == "nvfp4":
        return fm.nvfp4_fake_quant(w_e, axis=-1)      # 1x16 blocks along K, a global scale per row
    if precision == "mxfp8":
        if blocks == "1x32":
            return fm.mx_fake_quant(w_e, axis=-1)
        q, e = fm.mx_quantize_weight_32x32(w_e)
        return fm.mx_dequantize_weight_32x32(q, e)
    return w_e


def swiglu(g, u, limit=0.0):
    """h2 = SiLU(g) * u, with g clamped to <= limit and u to [-limit, limit]
    when limit > 0 (clamped SwiGLU, reading in the module docstring)."""
    if limit > 0:
        g = np.minimum(g, limit)
        u = np.clip(u, -limit, limit)
    return silu(g) * u


def swiglu_grad(g, u, dh, limit=0.0):
    """(dg, du) of ``swiglu`` at (g, u) for the upstream gradient dh."""
    if limit > 0:
        gc, uc = np.minimum(g, limit), np.clip(u, -limit, limit)
        return dh * uc * silu_grad(gc) * (g <= limit), dh * silu(gc) * (np.abs(u) <= limit)
    return dh * u * silu_grad(g), dh * silu(g)


def clip_counts(h1, F, limit):
    """Numbers of gate and up values the clamp changes (clip statistics)."""
    if limit <= 0:
        return 0, 0
    return int(np.sum(h1[:, :F] > limit)), int(np.sum(np.abs(h1[:, F:]) > limit))


# ------------------------------------------------------------------ forward

def forward(x, ids, scores, w13, w2, precision, out_init=None, pad=PAD, swiglu_limit=0.0, weight_blocks="32x32"):
    """Routed forward (see module docstring).

    x [T,D] (BF16 values as float64), ids [T,K] int, scores [T,K] float32,
    w13 [E,2F,D] and w2 [E,D,F] (anything indexable by expert returning BF16
    values).  ``out_init`` [T,D] is added before the final rounding (the
    accumulate mode used to add a shared expert).  Returns a dict with
    ``out`` and the saved state used by ``backward``.
    """
    assert precision in PRECISIONS
    x = np.asarray(x, dtype=np.float64)
    T, D = x.shape
    K = ids.shape[1]
    E = len(w13)
    F = np.asarray(w13[0]).shape[0] // 2
    rt = route(ids, E, pad)
    Rp = int(rt.poffsets[E])
    tok = np.where(rt.perm >= 0, rt.perm // K, -1)
    xg = np.zeros((Rp, D))
    xg[rt.perm >= 0] = x[tok[rt.perm >= 0]]
    xq = _q_row(xg, precision)
    h1 = np.zeros((Rp, 2 * F))
    h2 = np.zeros((Rp, F))
    h3 = np.zeros((Rp, D))
    h1_exact = np.zeros((Rp, 2 * F))
    for e in range(E):
        a, b = rt.poffsets[e], rt.poffsets[e + 1]
        if a == b:
            continue
        w13e = prepare_weight(w13[e], precision, weight_blocks)
        h1_exact[a:b] = xq[a:b] @ w13e.T
        h1[a:b] = _round_out(h1_exact[a:b], precision)
    g, u = h1[:, :F], h1[:, F:]
    h2 = swiglu(g, u, swiglu_limit)
    h2q = _q_row(h2, precision)
    for e in range(E):
        a, b = rt.poffsets[e], rt.poffsets[e + 1]
        if a == b:
            continue
        w2e = prepare_weight(w2[e], precision, weight_blocks)
        h3[a:b] = _round_out(h2q[a:b] @ w2e.T, precision)
    out = combine(h3, rt.inv.reshape(T, K), scores, out_init, precision)
    return dict(out=out, routing=rt, xg=xg, xq=xq, h1=h1, h1_exact=h1_exact, h2=h2, h2q=h2q,
                h3=h3, ids=np.asarray(ids), scores=np.asarray(scores, np.float32),
                precision=precision, T=T, D=D, F=F, E=E, K=K, swiglu_limit=swiglu_limit,
                clip=clip_counts(h1, F, swiglu_limit))


def combine(h3, inv, scores, out_init, precision):
    """out[t] = R(init[t] + sum_k s(t,k) h3[inv(t,k)]) over active routes
    (blog section 2 combine with index_add; Dist-MoE explainer section 01:
    the owner applies the scores and sums the K routes wide)."""
    T, K = inv.shape
    acc = np.zeros((T, h3.shape[1])) if out_init is None else np.array(out_init, np.float64)
    s = np.asarray(scores, dtype=np.float64)
    for k in range(K):
        on = inv[:, k] >= 0
        acc[on] += s[on, k, None] * h3[inv[on, k]]
    return _round_out(acc, precision)


# ----------------------------------------------------------------- backward

def backward(state, dY, w13, w2, dx_init=None, dw_fp32=False):
    """Backward of ``forward`` (see module docstring).

    Returns dict with dX [T,D], dp [T,K] (score gradient), dW13 [E,2F,D],
    dW2 [E,D,F] and the intermediates dh3/dh2/dh1/dxr per padded row.
    """
    p = state["precision"]
    assert p != "nvfp4", "NVFP4 is an inference format here (no backward)"
    rt = state["routing"]
    T, D, F, E, K = (state[k] for k in ("T", "D", "F", "E", "K"))
    Rp = int(rt.poffsets[E])
    dY = np.asarray(dY, dtype=np.float64)
    s32 = state["scores"].astype(np.float32).reshape(-1)
    dh3 = np.zeros((Rp, D))
    rows = rt.perm >= 0
    ridx = rt.perm[rows]
    if p == "f64":
        dh3[rows] = s32[ridx, None].astype(np.float64) * dY[ridx // K]
    else:
        dh3[rows] = (s32[ridx, None] * dY[ridx // K].astype(np.float32)).astype(np.float64)
    dh3_row = _q_row(dh3, p)
    dh3_col = _q_col(dh3, p)
    h1 = state["h1"]
    g, u = h1[:, :F], h1[:, F:]
    dh2 = np.zeros((Rp, F))
    for e in range(E):
        a, b = rt.poffsets[e], rt.poffsets[e + 1]
        if a == b:
            continue
        dh2[a:b] = dh3_row[a:b] @ prepare_weight(w2[e], p)
    dg, du = swiglu_grad(g, u, dh2, state.get("swiglu_limit", 0.0))
    dh1 = np.concatenate([dg, du], axis=1)
    dh1_row = _q_row(dh1, p)
    dh1_col = _q_col(dh1, p)
    h2_col = state["h2q"] if p != "mxfp8" else _q_col(state["h2"], p)
    x_col = state["xq"] if p != "mxfp8" else _q_col(state["xg"], p)
    dxr = np.zeros((Rp, D))
    dW13 = np.zeros((E, 2 * F, D))
    dW2 = np.zeros((E, D, F))
    for e in range(E):
        a, b = rt.poffsets[e], rt.poffsets[e + 1]
        if a == b:
            continue
        dxr[a:b] = _round_out(dh1_row[a:b] @ prepare_weight(w13[e], p), p)
        dW2[e] = dh3_col[a:b].T @ h2_col[a:b]
        dW13[e] = dh1_col[a:b].T @ x_col[a:b]
    if p != "f64":
        rw = fm.round_fp32 if dw_fp32 else fm.round_bf16
        dW2, dW13 = rw(dW2), rw(dW13)
    inv = rt.inv.reshape(T, K)
    acc = np.zeros((T, D)) if dx_init is None else np.array(dx_init, np.float64)
    for k in range(K):
        on = inv[:, k] >= 0
        acc[on] += dxr[inv[on, k]]
    dX = _round_out(acc, p)
    # score gradient dp(t,k) = <h3(t,k), dY[t]> (blog section 2, "SwiGLU
    # backward": the routing-weight gradient of the weighted combine); zero for
    # inactive routes
    dp = np.zeros((T, K))
    for k in range(K):
        on = inv[:, k] >= 0
        dp[on, k] = np.sum(state["h3"][inv[on, k]] * dY[on], axis=1)
    return dict(dX=dX, dp=dp, dW13=dW13, dW2=dW2, dh3=dh3, dh3_row=dh3_row,
                dh3_col=dh3_col, dh2=dh2, dh1=dh1, dh1_row=dh1_row,
                dh1_col=dh1_col, dxr=dxr, h2_col=h2_col, x_col=x_col)


# ------------------------------------------------- brute-force per-token forward

def forward_per_token(x, ids, scores, w13, w2, precision, out_init=None, tokens=None, swiglu_limit=0.0,
                      weight_blocks="32x32"):
    """Forward without any permutation: for each token, loop over its K
    routes and run that expert's SwiGLU FFN on the single row.

    Pins the routed ``forward`` (grouping, padding, inverse permutation and
    combine) and serves sampled checks at full size (``tokens`` selects the
    rows computed; weights are fetched one expert at a time)."""
    x = np.asarray(x, dtype=np.float64)
    T, D = x.shape
    K = ids.shape[1]
    E = len(w13)
    tokens = range(T) if tokens is None else tokens
    cache = {}

    def wts(e):
        if e not in cache:
            cache[e] = (prepare_weight(w13[e], precision, weight_blocks),
                        prepare_weight(w2[e], precision, weight_blocks))
        return cache[e]

    out = {}
    for t in tokens:
        acc = np.zeros(D) if out_init is None else np.array(out_init[t], np.float64)
        xt = _q_row(x[t][None, :], precision)[0]
        for k in range(K):
            e = int(ids[t, k])
            if e < 0 or e >= E:
                continue
            w13e, w2e = wts(e)
            F = w13e.shape[0] // 2
            h1 = _round_out(w13e @ xt, precision)
            h2 = _q_row(swiglu(h1[:F], h1[F:], swiglu_limit)[None, :], precision)[0]
            h3 = _round_out(w2e @ h2, precision)
            acc = acc + np.float64(np.float32(scores[t, k])) * h3
        out[t] = _round_out(acc, precision)
    return out
