"""NVFP4 inference on the GPU against the oracle.

* Weight preparation: codes, block scales and row scales of every row equal
  the oracle's quantiser (``oracle.formats.nvfp4_quantize``) value for value,
  on rows built to reach its corners (a zero row, a zero block, a dominant
  value, block scales down to the E4M3 subnormals) and on the hand-worked
  rows of ``golden/nvfp4_hand_blocks.json``.
* The routed x rows the forward quantises into its routing blocks equal the
  oracle's quantisation of the gathered rows, bit for bit; the h2 rows,
  decided from FP32 values that both sides form in a different order, agree
  on all but a few codes.
* The forward: out within TOL["nvfp4"] of the oracle's NVFP4 forward on
  small ragged cases (several 128-row blocks, 32-row remainders, inactive
  routes, a clamped SwiGLU, accumulation onto an existing out), at the
  E=384, D=7168 inference shape on sampled tokens, and at one token; a
  call whose routes are all inactive gives exact zeros, and T = 0 enqueues
  nothing.
"""

import json
import os

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth
from oracle import formats as fm
from oracle import sample as osample

from moe_cases import TOL, Case, assert_routing, ctx_routing, rel_err, run_gpu, run_oracle, to_f64

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_hand_blocks.json")


def decode_chunks(raw, row_tiles, K):
    """Chunks of 128 rows x 64 values (4096 code bytes, then 512 scale
    bytes) -> E2M1 values [row_tiles * 128, K] and E4M3 block scales
    [row_tiles * 128, K / 16], as float64."""
    ks = K // 64
    c = np.asarray(raw, dtype=np.uint8)[: row_tiles * ks * 4608].reshape(row_tiles, ks, 4608)
    codes = c[:, :, :4096].reshape(row_tiles, ks, 128, 32)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(row_tiles, ks, 128, 64)
    q = fm.e2m1_decode(nib).transpose(0, 2, 1, 3).reshape(row_tiles * 128, K)
    sc = c[:, :, 4096:].reshape(row_tiles, ks, 128, 4)
    sb = fm.e4m3_decode(sc).transpose(0, 2, 1, 3).reshape(row_tiles * 128, K // 16)
    return q, sb


def _structured_weight(E, N, K, rng):
    w = rng.standard_normal((E, N, K)) / np.sqrt(K)
    ramp = np.repeat(2.0 ** -np.arange(K // 16, dtype=np.float64), 16)
    w[0, 5] = np.abs(w[0, 5]) * ramp          # block maxima 2^0 .. 2^-(K/16-1): subnormal and zero scales
    w[0, 7] = 0.0                             # zero row
    w[1, 3, 16:32] = 0.0                      # a zero block in a live row
    w[1, 9, 0] = 1.0e4                        # one dominant value: the other blocks get small scales
    golden = json.load(open(GOLDEN))["rows"]
    for i, row in enumerate(golden):
        w[1, 100 + i] = 0.0
        w[1, 100 + i, : len(row["values"])] = row["values"]
    return torch.from_numpy(w).to(torch.bfloat16), golden


def test_weight_prep_matches_oracle_and_hand_worked_rows():
    from mixture_experts_routed_route_gb300.layer import PreparedWeight
    E, N, K = 2, 256, 512
    wb, golden = _structured_weight(E, N, K, np.random.default_rng(11))
    W = PreparedWeight(wb.cuda(), "nvfp4", with_transpose=False)
    torch.cuda.synchronize()
    q, sb = decode_chunks(W.data.cpu().numpy(), E * N // 128, K)
    g = W.scale.cpu().numpy().astype(np.float64)
    oq, osb, og = fm.nvfp4_quantize(to_f64(wb).reshape(E * N, K), axis=-1)
    assert np.array_equal(g, og)
    assert np.array_equal(sb, osb)
    assert np.array_equal(q, oq)
    assert np.all(q[7] == 0) and g[7] == 0.0            # the zero row
    assert np.min(sb[5][sb[5] > 0]) < 2.0 ** -6         # E4M3 subnormal block scales were reached
    for i, row in enumerate(golden):
        r = N + 100 + i
        n = len(row["values"])
        assert g[r] == row["g"], row["name"]
        assert np.array_equal(sb[r, : n // 16], row["block_scales"]), row["name"]
        assert np.array_equal(q[r, :n], row["q"]), row["name"]


def _f4_small(name, seed, **kw):
    base = dict(T=160, D=256, F=384, E=6, K=3, precision="nvfp4", routing="zipf", inactive_frac=0.1, zipf_s=1.3)
    base.update(kw)
    return synth.Workload(name, seed=seed, **base)


SMALL = {
    "zipf": lambda: _f4_small("f4_a", 41),
    "uniform_wide": lambda: _f4_small("f4_b", 42, D=512, F=256, E=10, K=2, routing="uniform"),
    "long_k": lambda: _f4_small("f4_c", 43, T=96, D=1024, F=640, E=4, K=2, routing="uniform"),
}


def _routing_blocks(layer):
    from mixture_experts_routed_route_gb300 import abi
    _, nbytes = abi.moe_ctx_buffer(layer.ctx, abi.MOE_BUF_ROUTING)
    raw = layer.read_buffer(abi.MOE_BUF_ROUTING, np.uint8, (nbytes,))
    hdr_off, _ = abi.moe_saved_state_field(layer.cfg, abi.MOE_SAVED_HEADER)
    nblk = int(raw[hdr_off:hdr_off + 16].view(np.int32)[1])
    off, _ = abi.moe_saved_state_field(layer.cfg, abi.MOE_SAVED_BLOCKS)
    return raw[off:off + 16 * nblk].view(np.int32).reshape(nblk, 4)


def _routed_rows(layer, which_chunks, which_g, K, rows_total):
    """Decode a context's routed-row chunks back to row order."""
    from mixture_experts_routed_route_gb300 import abi
    blocks = _routing_blocks(layer)
    _, nbytes = abi.moe_ctx_buffer(layer.ctx, which_chunks)
    raw = layer.read_buffer(which_chunks, np.uint8, (nbytes,))
    q, sb = decode_chunks(raw, len(blocks), K)
    g = layer.read_buffer(which_g, np.float32, (rows_total,)).astype(np.float64)
    rq = np.zeros((rows_total, K))
    rsb = np.zeros((rows_total, K // 16))
    for b, (e, r0, n, _) in enumerate(blocks):
        rq[r0:r0 + n] = q[128 * b:128 * b + n]
        rsb[r0:r0 + n] = sb[128 * b:128 * b + n]
    return rq, rsb, g


@pytest.mark.parametrize("name", list(SMALL))
def test_small_forward_matches_oracle(name):
    from mixture_experts_routed_route_gb300 import abi
    case = Case(SMALL[name]())
    w = case.w
    g = run_gpu(case, training=False, backward=False)
    assert g["err_bits"] == 0
    layer = g["layer"]
    assert_routing(ctx_routing(layer, case.T), case.ids.astype(np.int64), w.E)
    o = run_oracle(case, backward=False)
    st = o["state"]
    Rp = int(st["routing"].poffsets[w.E])

    # x rows: identical codes, block scales and row scales
    xq, xsb, xg = _routed_rows(layer, abi.MOE_BUF_XROW, abi.MOE_BUF_XROW_SCALE, w.D, Rp)
    oq, osb, og = fm.nvfp4_quantize(st["xg"], axis=-1)
    assert np.array_equal(xg, og) and np.array_equal(xsb, osb) and np.array_equal(xq, oq)

    # h2: the FP32 values the quantiser saw, then the codes
    h2 = layer.read_buffer(abi.MOE_BUF_H2F, np.float32, (Rp, w.F)).astype(np.float64)
    assert rel_err(h2, st["h2"]) <= 1e-2
    hq, hsb, hg = _routed_rows(layer, abi.MOE_BUF_H2ROW, abi.MOE_BUF_H2ROW_SCALE, w.F, Rp)
    oq2, osb2, og2 = fm.nvfp4_quantize(fm.round_fp32(st["h2"]), axis=-1)
    assert np.mean(hq != oq2) <= 1e-3
    assert np.mean(hsb != osb2) <= 1e-3

    assert rel_err(g["out"], o["out"]) <= TOL["nvfp4"]
    dead = np.all(case.ids < 0, axis=1)
    assert np.all(g["out"][dead] == 0.0)
    layer.close()


def test_clamped_swiglu_forward_matches_oracle():
    case = Case(SMALL["zipf"]())
    lim = 0.75
    g = run_gpu(case, training=False, backward=False, swiglu_limit=lim)
    assert g["err_bits"] == 0
    o = run_oracle(case, backward=False, swiglu_limit=lim)
    assert rel_err(g["out"], o["out"]) <= TOL["nvfp4"]
    gate, up = o["state"]["clip"]
    assert gate + up > 0                           # the limit is active in this case
    assert tuple(g["layer"].clip_stats()) == (gate, up)
    g["layer"].close()


def _sampled_parity(w, T, tokens_wanted, seed):
    from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight
    dev = torch.device("cuda")
    D, F, E, K = w.D, w.F, w.E, w.K
    ids, scores = synth.make_routing(w)
    ids, scores = ids[:T], scores[:T]
    x = synth.make_tokens(w, dev)[:T].contiguous()
    w13, w2 = synth.make_weights(w, dev)
    W13 = PreparedWeight(w13, "nvfp4", with_transpose=False)
    W2 = PreparedWeight(w2, "nvfp4", with_transpose=False)
    layer = MoELayer(T, D, F, E, K, "nvfp4", training=False)
    out = layer.forward(x, torch.from_numpy(ids).to(dev), torch.from_numpy(scores).to(dev), W13, W2)
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    assert_routing(ctx_routing(layer, T), ids.astype(np.int64), E)
    rng = np.random.default_rng(seed)
    tokens = sorted(rng.choice(T, size=min(tokens_wanted, T), replace=False).tolist())
    experts = sorted(set(int(e) for t in tokens for e in ids[t] if e >= 0))
    st = osample.run(to_f64(x), ids, scores, to_f64(w13[experts]), to_f64(w2[experts]), experts, "nvfp4")
    assert rel_err(to_f64(out[tokens]), st["out"][tokens]) <= TOL["nvfp4"]
    layer.close()


def test_e384_inference_shape_sampled_tokens():
    """T=2048, D=7168, F=2048, E=384, K=6, uniform routing (the MXFP8
    inference configuration's routed layer, here in NVFP4)."""
    _sampled_parity(synth.WORKLOADS["e384_nvfp4"], 2048, 4, 78)


def test_one_token_at_the_e384_shape():
    _sampled_parity(synth.WORKLOADS["e384_nvfp4"], 1, 1, 79)


def test_inactive_routes_accumulate_and_empty_calls():
    """Every route inactive: no routing block, so both GEMMs have no tile and
    out is exactly zero (or the accumulated input, rounded once).  With
    MOE_ACCUMULATE_OUT on a live case, out_init is added before the single
    rounding, as the oracle does.  T = 0 enqueues nothing."""
    case = Case(SMALL["zipf"]())
    dead = Case(SMALL["zipf"](), ids=np.full_like(case.ids, -1), scores=np.zeros_like(case.scores))
    g = run_gpu(dead, training=False, backward=False)
    assert g["err_bits"] == 0 and np.all(g["out"] == 0.0)
    g["layer"].close()
    init = torch.randn((case.T, case.w.D), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    g = run_gpu(case, training=False, backward=False, out_init=init.cuda())
    assert g["err_bits"] == 0
    o = run_oracle(case, backward=False, out_init=to_f64(init))
    assert rel_err(g["out"], o["out"]) <= TOL["nvfp4"]
    layer, W13, W2 = g["layer"], g["W13"], g["W2"]
    dev = torch.device("cuda")
    empty = torch.empty((0, case.w.D), dtype=torch.bfloat16, device=dev)
    layer.forward(empty, torch.empty((0, case.w.K), dtype=torch.int32, device=dev),
                  torch.empty((0, case.w.K), dtype=torch.float32, device=dev), W13, W2, out=empty)
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    layer.close()


@pytest.mark.parametrize("name", ["zipf", "long_k"])
def test_few_ctas_walk_many_tiles_bit_for_bit(name):
    """With the persistent grids capped at 1 and 3 CTAs each CTA walks every
    or every third tile, through both accumulator buffers and many passes of
    the staging and operand rings; the output equals the uncapped run's bit
    for bit (a tile's K sum does not depend on which CTA runs it)."""
    case = Case(SMALL[name]())
    ref = run_gpu(case, training=False, backward=False)
    ref["layer"].close()
    for ctas in (1, 3):
        g = run_gpu(case, training=False, backward=False, max_ctas=ctas)
        assert g["err_bits"] == 0
        assert np.array_equal(g["out"], ref["out"]), ctas
        g["layer"].close()
