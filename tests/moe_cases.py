"""Shared helpers of the parity tests: seeded cases, the CUDA path through the
C ABI, and the oracle on the same inputs.

Inputs come from the seeded generator only; expected values come from the
oracle only.
"""

import numpy as np
import torch

from mixture_experts_routed_route_gb300 import synth

# max|gpu - ref| / max|ref|.  NVFP4 takes the MXFP8 bound: both sides
# quantise the same FP32 values with the same FP32 steps, so the operands are
# the same codes except where the two accumulation orders move an FP32 value
# across a rounding boundary.
TOL = {"bf16": 1e-2, "mxfp8": 3e-2, "nvfp4": 3e-2}


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / den)


def to_f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def bf16_from_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


class Case:
    """One seeded workload: inputs on the CPU (torch) and their fp64 copies."""

    def __init__(self, w, T=None, ids=None, scores=None, seed_layer=0):
        self.w = w
        self.T = w.T if T is None else T
        if ids is None:
            ids, scores = synth.make_routing(w, layer=seed_layer)
        self.ids = np.ascontiguousarray(ids[: self.T]).astype(np.int32)
        self.scores = np.ascontiguousarray(scores[: self.T]).astype(np.float32)
        self.x = synth.make_tokens(w, "cpu", layer=seed_layer)[: self.T].contiguous()
        self.dy = synth.make_grad_out(w, "cpu", layer=seed_layer)[: self.T].contiguous()
        self.w13, self.w2 = synth.make_weights(w, "cpu", layer=seed_layer)

    # fp64 views for the oracle
    def oracle_inputs(self):
        return (to_f64(self.x), self.ids.astype(np.int64), self.scores, to_f64(self.w13), to_f64(self.w2))


def run_gpu(case, precision=None, training=True, debug=False, out_init=None, max_tokens=None,
            dx_init=None, dw_fp32=False, backward=True, swiglu_limit=0.0, weight_prec=None, max_ctas=0,
            tile_mode=0, mn_major=False):
    """Forward (and backward) of a case through the C ABI; returns a dict of
    host arrays plus the layer object for further inspection.  weight_prec
    overrides the weights' preparation (e.g. "mxfp8_1x32"); max_ctas caps
    the persistent grids (moe_ctx_set_max_ctas); tile_mode picks the
    grouped GEMMs' B tiles (moe_ctx_test_tile_mode: 1 row blocks, 2
    row-block pairs, 0 the context's default); mn_major: MXFP8 weights
    without transposed codes."""
    from mixture_experts_routed_route_gb300 import abi
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight

    w = case.w
    precision = precision or w.precision
    dev = torch.device("cuda")
    T = case.T
    layer = MoELayer(max_tokens or max(T, 1), w.D, w.F, w.E, w.K, precision, training=training, debug=debug,
                     swiglu_limit=swiglu_limit)
    if max_ctas:
        abi.moe_ctx_set_max_ctas(layer.ctx, max_ctas)
    if tile_mode:
        abi.moe_ctx_test_tile_mode(layer.ctx, tile_mode)
    W13 = PreparedWeight(case.w13.to(dev), weight_prec or precision, with_transpose=training, mn_major=mn_major)
    W2 = PreparedWeight(case.w2.to(dev), weight_prec or precision, with_transpose=training, mn_major=mn_major)
    x = case.x.to(dev)
    ids = torch.from_numpy(case.ids).to(dev)
    sc = torch.from_numpy(case.scores).to(dev)
    out = torch.zeros((T, w.D), dtype=torch.bfloat16, device=dev)
    acc = out_init is not None
    if acc:
        out.copy_(out_init)
    saved = layer.new_saved() if training else None
    layer.forward(x, ids, sc, W13, W2, out=out, saved=saved, accumulate=acc)
    res = {"layer": layer, "W13": W13, "W2": W2, "saved": saved, "out": to_f64(out), "out_t": out}
    if training and backward:
        dy = case.dy.to(dev)
        dx = torch.zeros((T, w.D), dtype=torch.bfloat16, device=dev)
        if dx_init is not None:
            dx.copy_(dx_init)
        dp = torch.full((T, w.K), float("nan"), dtype=torch.float32, device=dev)
        dx, dW13, dW2 = layer.backward(saved, dy, W13, W2, dx=dx, accumulate_dx=dx_init is not None,
                                       dw_fp32=dw_fp32, d_scores=dp)
        res.update(dx=to_f64(dx), dW13=to_f64(dW13), dW2=to_f64(dW2), dp=to_f64(dp))
    torch.cuda.synchronize()
    res["err_bits"] = layer.error_bits()
    return res


def run_oracle(case, precision=None, out_init=None, dx_init=None, dw_fp32=False, backward=True, swiglu_limit=0.0,
               weight_blocks="32x32"):
    from oracle import moe
    precision = precision or case.w.precision
    x, ids, s, w13, w2 = case.oracle_inputs()
    st = moe.forward(x, ids, s, w13, w2, precision, out_init=out_init, swiglu_limit=swiglu_limit,
                     weight_blocks=weight_blocks)
    res = {"state": st, "out": st["out"]}
    if backward:
        g = moe.backward(st, to_f64(case.dy), w13, w2, dx_init=dx_init, dw_fp32=dw_fp32)
        res.update(dx=g["dX"], dW13=g["dW13"], dW2=g["dW2"], dp=g["dp"], grads=g)
    return res


def ctx_routing(layer, T):
    """Routing arrays of the last inference forward (the context's copy,
    laid out like the routing prefix of a saved state)."""
    from mixture_experts_routed_route_gb300 import abi
    _, nbytes = abi.moe_ctx_buffer(layer.ctx, abi.MOE_BUF_ROUTING)
    raw = layer.read_buffer(abi.MOE_BUF_ROUTING, np.uint8, (nbytes,))

    def field(f, n):
        off, _ = abi.moe_saved_state_field(layer.cfg, f)
        return raw[off:off + 4 * n].view(np.int32)

    hdr = field(abi.MOE_SAVED_HEADER, 16)
    return {"hdr": hdr, "counts": field(abi.MOE_SAVED_COUNTS, layer.E),
            "poffsets": field(abi.MOE_SAVED_POFFSETS, layer.E + 1), "perm": field(abi.MOE_SAVED_PERM, int(hdr[2])),
            "inv": field(abi.MOE_SAVED_INV, T * layer.K)}


def assert_routing(got, ids, E):
    from oracle import moe as omoe
    rt = omoe.route(ids, E)
    assert got["hdr"][0] == ids.shape[0] and got["hdr"][2] == rt.poffsets[-1] and got["hdr"][3] == rt.num_active
    np.testing.assert_array_equal(got["counts"], rt.counts)
    np.testing.assert_array_equal(got["poffsets"], rt.poffsets)
    np.testing.assert_array_equal(got["perm"], rt.perm)
    np.testing.assert_array_equal(got["inv"], rt.inv)


# ------------------------------------------------------------------------
# MXFP8 weight gradients: codes that two correct computations may round
# differently.
#
# The WGRAD operands h2 and dh1 are quantised (along rows, 32-row blocks)
# from values each side computes in its own precision: the GPU accumulates
# the GEMM in FP32, the oracle exactly.  Where such a value lies within the
# FP32 spread of a rounding decision (an E4M3 midpoint, a block-scale power
# of two, or the BF16 rounding of the h1 it is built from), both codes are
# correct, and one differing code moves a whole dW row by one E4M3 step.
# The check below compares what is unique with the stated tolerance and
# allows, on top of it, exactly the contribution of the undecided codes, all
# derived from oracle values.  EPS_ACC = 3 sqrt(K) 2^-24 for K = 7168 (the
# relative spread of an FP32 sum of K random-sign terms, three sigma).

EPS_ACC = 2.0 ** -16


def _bf16_candidates(v_exact, eps):
    """BF16 rounding of each exact value, and the other neighbour where the
    exact value lies within eps (relative) of a rounding midpoint."""
    from oracle import formats as fm
    r = fm.round_bf16(v_exact)
    lo = fm.round_bf16(v_exact * (1 - eps))
    hi = fm.round_bf16(v_exact * (1 + eps))
    return r, np.where(lo != r, lo, np.where(hi != r, hi, r))


def _mx_col_spread(cands, eps):
    """Per element, the spread of the dequantised MXFP8 column-bundle value
    over the admissible pre-quantisation values (each candidate scaled by
    1 - eps, 1, 1 + eps); zero where the code is decided."""
    from oracle import formats as fm
    lo = hi = None
    for c in cands:
        for f in (1 - eps, 1.0, 1 + eps):
            q = fm.mx_fake_quant(c * f, axis=0)
            lo = q if lo is None else np.minimum(lo, q)
            hi = q if hi is None else np.maximum(hi, q)
    return hi - lo


def mx_wgrad_allowance(state, grads, i):
    """(allow13, allow2, undecided13, undecided2) of oracle expert i: the
    per-element allowance on top of the tolerance for dW13 and dW2 (twice
    the spread of the undecided column-bundle codes times the other
    operand's magnitudes), and the fractions of undecided codes in the dh1
    and h2 column bundles.  Zero arrays for an expert without rows."""
    from oracle import moe as omoe
    rt = state["routing"]
    F = state["F"]
    a, b = int(rt.poffsets[i]), int(rt.poffsets[i + 1])
    if a == b:
        return np.zeros_like(grads["dW13"][i]), np.zeros_like(grads["dW2"][i]), 0.0, 0.0
    h1x = state["h1_exact"][a:b]
    g, ga = _bf16_candidates(h1x[:, :F], EPS_ACC)
    u, ua = _bf16_candidates(h1x[:, F:], EPS_ACC)
    dh2 = grads["dh2"][a:b]
    lim = state.get("swiglu_limit", 0.0)
    combos = [(g, u), (ga, u), (g, ua), (ga, ua)]
    dh1_c = [np.concatenate(omoe.swiglu_grad(gg, uu, dh2, lim), axis=1) for gg, uu in combos]
    h2_c = [omoe.swiglu(gg, uu, lim) for gg, uu in combos]
    s13 = _mx_col_spread(dh1_c, EPS_ACC)
    s2 = _mx_col_spread(h2_c, EPS_ACC)
    allow13 = 2.0 * s13.T @ np.abs(grads["x_col"][a:b])
    allow2 = 2.0 * np.abs(grads["dh3_col"][a:b]).T @ s2
    return allow13, allow2, float((s13 > 0).mean()), float((s2 > 0).mean())


def check_mx_wgrad(dW13_gpu, dW2_gpu, state, grads, experts=None, tol=TOL["mxfp8"], max_undecided=5e-3):
    """Assert dW13/dW2 of the listed experts (indices into the oracle's
    expert axis; dW*_gpu indexed the same way) against the oracle with the
    undecided-code allowance.  Returns the per-expert plain errors."""
    rt = state["routing"]
    experts = range(len(grads["dW13"])) if experts is None else experts
    errs = []
    for i in experts:
        a, b = int(rt.poffsets[i]), int(rt.poffsets[i + 1])
        ref13, ref2 = grads["dW13"][i], grads["dW2"][i]
        got13, got2 = np.asarray(dW13_gpu[i], np.float64), np.asarray(dW2_gpu[i], np.float64)
        if a == b:
            assert np.all(got13 == 0) and np.all(got2 == 0)
            errs.append((0.0, 0.0))
            continue
        allow13, allow2, u13, u2 = mx_wgrad_allowance(state, grads, i)
        assert u13 <= max_undecided and u2 <= max_undecided
        for got, ref, allow, name in ((got13, ref13, allow13, "dW13"), (got2, ref2, allow2, "dW2")):
            bound = tol * np.max(np.abs(ref)) + allow
            bad = np.abs(got - ref) > bound
            assert not bad.any(), (name, i, int(bad.sum()), rel_err(got, ref))
        errs.append((rel_err(got13, ref13), rel_err(got2, ref2)))
    return errs


# ------------------------------------------------------------------------
# MXFP8 scale layouts (include/moe_gb300.h): 512-byte atoms of 128 rows x 4
# consecutive 32-value blocks, row p / block l at byte (p%32)*16 + (p//32)*4 + l.

def atom_byte(p, l):
    return (p % 32) * 16 + (p // 32) * 4 + l


def unpack_row_sf(atoms, blocks, rows, K):
    """[rows, K/32] scale bytes of a row bundle stored as atoms [B_cap][K/128]."""
    atoms = np.asarray(atoms).reshape(-1)
    out = np.zeros((rows, K // 32), np.uint8)
    kb = np.arange(K // 32)[None, :]
    for b, (_, r0, n, _) in enumerate(np.asarray(blocks).reshape(-1, 4)):
        p = np.arange(n)[:, None]
        out[r0:r0 + n] = atoms[(b * (K // 128) + kb // 4) * 512 + atom_byte(p, kb % 4)]
    return out


def unpack_col_sf(atoms, blocks, dim, rows, b_cap):
    """[dim, rows/32] scale bytes of a column bundle stored as atoms [dim/128][B_cap]."""
    atoms = np.asarray(atoms).reshape(-1)
    out = np.zeros((dim, rows // 32), np.uint8)
    d = np.arange(dim)
    for b, (_, r0, n, _) in enumerate(np.asarray(blocks).reshape(-1, 4)):
        for l in range(n // 32):
            out[:, r0 // 32 + l] = atoms[((d // 128) * b_cap + b) * 512 + atom_byte(d % 128, l)]
    return out


def unpack_weight_sf(atoms, rows, K):
    """[rows, K/32] scale bytes of a weight stored as atoms [rows/128][K/128]."""
    atoms = np.asarray(atoms).reshape(-1)
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 32)[None, :]
    return atoms[((r // 128) * (K // 128) + kb // 4) * 512 + atom_byte(r % 128, kb % 4)]


def saved_blocks(layer, saved):
    """Row blocks (expert, first row, rows, 0) of the routing in `saved`."""
    from mixture_experts_routed_route_gb300 import abi
    hdr = layer.saved_field(saved, abi.MOE_SAVED_HEADER, torch.int32, (16,)).cpu().numpy()
    nb = int(hdr[1])
    return layer.saved_field(saved, abi.MOE_SAVED_BLOCKS, torch.int32, (4 * nb,)).cpu().numpy().reshape(nb, 4)
