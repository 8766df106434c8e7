"""Pins of the MXFP8 weight-gradient parity check (``moe_cases.check_mx_wgrad``).

The weight-gradient operands h2 and dh1 are quantised from values each side
computes at its own precision, so the check adds to the stated tolerance the
contribution of codes that lie on a rounding decision ("Dist-MoE:
Speed-of-light distributed Mixture-of-Experts kernels", section 02,
"Quantization Axes for Forward and Backward": the column bundles are
quantised along the rows the weight gradient contracts over).  These tests
hold that allowance to account, on the CPU, with oracle values only:

* it accepts the oracle against itself, and a recomputation of the weight
  gradients from inputs that a correct FP32 pipeline may produce (h1 moved
  inside the FP32 accumulation spread before its BF16 rounding, h2 and dh2
  moved by a few FP32 ulps);
* it rejects planted errors: one element moved by twice the tolerance, one
  decided column-bundle code with its sign flipped, one row scaled by 1.05,
  and two experts' gradients swapped;
* its allowance stays small at the 384-expert, D=7168 shape: a stated bound
  on its mean over each sampled expert's gradient and on the share of
  elements it touches.
"""

import numpy as np
import pytest

from mixture_experts_routed_route_gb300 import synth
from oracle import formats as fm
from oracle import moe as omoe
from oracle import sample as osample

from moe_cases import EPS_ACC, TOL, Case, _mx_col_spread, check_mx_wgrad, mx_wgrad_allowance, run_oracle, to_f64

TOLMX = TOL["mxfp8"]


@pytest.fixture(scope="module")
def small():
    w = synth.Workload("chk", 192, 256, 256, 4, 2, "mxfp8", "zipf", inactive_frac=0.1, zipf_s=1.0, seed=41)
    case = Case(w)
    o = run_oracle(case)
    return case, o["state"], o["grads"]


def _wgrads_from(state, grads, h1, h2, dh2):
    """dW13, dW2 recomputed (as the oracle does) from given h1 (BF16), h2
    and dh2: column bundles quantised along rows, products in fp64, BF16
    result."""
    rt = state["routing"]
    E, F = state["E"], state["F"]
    lim = state.get("swiglu_limit", 0.0)
    dg, du = omoe.swiglu_grad(h1[:, :F], h1[:, F:], dh2, lim)
    dh1_col = fm.mx_fake_quant(np.concatenate([dg, du], axis=1), axis=0)
    h2_col = fm.mx_fake_quant(h2, axis=0)
    dW13 = np.zeros_like(grads["dW13"])
    dW2 = np.zeros_like(grads["dW2"])
    for e in range(E):
        a, b = int(rt.poffsets[e]), int(rt.poffsets[e + 1])
        if a == b:
            continue
        dW13[e] = dh1_col[a:b].T @ grads["x_col"][a:b]
        dW2[e] = grads["dh3_col"][a:b].T @ h2_col[a:b]
    return fm.round_bf16(dW13), fm.round_bf16(dW2)


def test_accepts_the_oracle_itself(small):
    _, st, gr = small
    errs = check_mx_wgrad(gr["dW13"], gr["dW2"], st, gr)
    assert all(e == (0.0, 0.0) for e in errs)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_accepts_an_admissible_fp32_recomputation(small, seed):
    """h1 before its BF16 rounding moved within half the accumulation spread,
    h2 and dh2 by up to 4 FP32 ulps: codes may change only where the
    allowance is nonzero, and the check must accept the result."""
    _, st, gr = small
    rng = np.random.default_rng(seed)
    h1x = st["h1_exact"]
    h1 = fm.round_bf16(h1x * (1 + rng.uniform(-0.5, 0.5, h1x.shape) * EPS_ACC))
    F = st["F"]
    h2 = omoe.swiglu(h1[:, :F], h1[:, F:], st.get("swiglu_limit", 0.0))
    h2 = h2 * (1 + rng.uniform(-4, 4, h2.shape) * 2.0 ** -24)
    dh2 = gr["dh2"] * (1 + rng.uniform(-4, 4, gr["dh2"].shape) * 2.0 ** -24)
    dW13, dW2 = _wgrads_from(st, gr, h1, h2, dh2)
    check_mx_wgrad(dW13, dW2, st, gr)
    # the recomputation did change codes somewhere (else this test shows nothing)
    changed = sum(int(np.sum(dW13[e] != gr["dW13"][e])) + int(np.sum(dW2[e] != gr["dW2"][e]))
                  for e in range(st["E"]))
    assert changed > 0


def _busiest(st):
    return int(np.argmax(np.diff(st["routing"].poffsets)))


@pytest.mark.parametrize("which", ["dW13", "dW2"])
def test_rejects_one_element_moved_by_twice_the_tolerance(small, which):
    _, st, gr = small
    i = _busiest(st)
    a13, a2, _, _ = mx_wgrad_allowance(st, gr, i)
    allow = a13 if which == "dW13" else a2
    ref = gr[which][i]
    pos = np.unravel_index(np.argmin(allow), allow.shape)
    assert allow[pos] < TOLMX * np.max(np.abs(ref))   # a position the allowance does not cover
    got = {k: gr[k].copy() for k in ("dW13", "dW2")}
    got[which][i][pos] += 2 * TOLMX * np.max(np.abs(ref))
    with pytest.raises(AssertionError):
        check_mx_wgrad(got["dW13"], got["dW2"], st, gr)


@pytest.mark.parametrize("which", ["h2", "dh1"])
def test_rejects_a_flipped_decided_column_code(small, which):
    """One code of a column bundle, at a position whose rounding is decided
    (zero spread), takes the opposite sign: the gradient of a kernel that
    wrote a wrong code there must fail."""
    _, st, gr = small
    i = _busiest(st)
    rt = st["routing"]
    a, b = int(rt.poffsets[i]), int(rt.poffsets[i + 1])
    F = st["F"]
    h1 = st["h1"]
    lim = st.get("swiglu_limit", 0.0)
    if which == "h2":
        col = fm.mx_fake_quant(st["h2"], axis=0)[a:b].copy()
        spread = _mx_col_spread([st["h2"][a:b]], EPS_ACC)
        other = gr["dh3_col"][a:b]
    else:
        dg, du = omoe.swiglu_grad(h1[:, :F], h1[:, F:], gr["dh2"], lim)
        raw = np.concatenate([dg, du], axis=1)
        col = fm.mx_fake_quant(raw, axis=0)[a:b].copy()
        spread = _mx_col_spread([raw[a:b]], EPS_ACC)
        other = gr["x_col"][a:b]
    # the decided code whose flip moves the gradient most
    weight = np.abs(col) * np.max(np.abs(other), axis=1)[:, None]
    weight[spread > 0] = -1
    r, f = np.unravel_index(np.argmax(weight), weight.shape)
    col[r, f] = -col[r, f]
    got13, got2 = gr["dW13"].copy(), gr["dW2"].copy()
    if which == "h2":
        got2[i] = fm.round_bf16(other.T @ col)
    else:
        got13[i] = fm.round_bf16(col.T @ other)
    with pytest.raises(AssertionError):
        check_mx_wgrad(got13, got2, st, gr)


@pytest.mark.parametrize("which", ["dW13", "dW2"])
def test_rejects_a_row_scaled_by_five_percent(small, which):
    _, st, gr = small
    i = _busiest(st)
    got = {k: gr[k].copy() for k in ("dW13", "dW2")}
    ref = gr[which][i]
    row = np.unravel_index(np.argmax(np.abs(ref)), ref.shape)[0]
    got[which][i][row] *= 1.05
    with pytest.raises(AssertionError):
        check_mx_wgrad(got["dW13"], got["dW2"], st, gr)


@pytest.mark.parametrize("which", ["dW13", "dW2"])
def test_rejects_two_experts_swapped(small, which):
    _, st, gr = small
    got = {k: gr[k].copy() for k in ("dW13", "dW2")}
    got[which][[0, 1]] = got[which][[1, 0]]
    with pytest.raises(AssertionError):
        check_mx_wgrad(got["dW13"], got["dW2"], st, gr)


def test_allowance_is_small_at_the_e384_shape():
    """At T=2048, D=7168, F=2048, E=384, K=6 (Zipf 1.2, 10 % inactive), for
    an expert of median load and one of heavy load: the allowance averages
    under 1/200 of the tolerance band, touches under 5 % of the elements,
    and under 1/200 of the column-bundle codes are undecided."""
    w = synth.WORKLOADS["e384_mxfp8_zipf_train"]
    ids, scores = synth.make_routing(w)
    cnt = np.bincount(ids[ids >= 0], minlength=w.E)
    order = np.argsort(cnt, kind="stable")
    experts = [int(order[w.E // 2]), int(order[int(0.885 * w.E)])]   # about 6 and 36 rows
    x = to_f64(synth.make_tokens(w, "cpu"))
    dy = to_f64(synth.make_grad_out(w, "cpu"))
    w13, w2 = synth.make_weights(w, "cpu", experts=experts)
    res = osample.run(x, ids, scores, to_f64(w13), to_f64(w2), experts, "mxfp8", dY=dy)
    st, gr = res["state"], res["grads"]
    for i in range(len(experts)):
        a13, a2, u13, u2 = mx_wgrad_allowance(st, gr, i)
        assert u13 <= 5e-3 and u2 <= 5e-3
        for allow, ref in ((a13, gr["dW13"][i]), (a2, gr["dW2"][i])):
            band = TOLMX * np.max(np.abs(ref))
            assert np.mean(allow) / band < 5e-3
            assert np.mean(allow > 0) < 0.05
