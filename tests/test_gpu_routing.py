"""F0 routing on the GPU against the oracle: counts, offsets, padded offsets,
permutation, inverse permutation, scores copy and row blocks, bit-exact."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_route_gb300 import synth
from oracle import moe as omoe

from moe_cases import Case, run_gpu

pytestmark = pytest.mark.gpu


def _routing_case(name):
    if name == "tiny":
        return Case(synth.WORKLOADS["tiny_bf16"])
    if name == "skewed":
        w = synth.Workload("skewed", 300, 128, 128, 16, 4, "bf16", "zipf", inactive_frac=0.1, zipf_s=1.5, seed=7)
        return Case(w)
    if name == "bad_ids":
        w = synth.Workload("bad", 64, 128, 128, 8, 3, "bf16", "uniform", seed=8)
        ids, s = synth.make_routing(w)
        ids[3, :] = -1
        s[3, :] = 0.0
        ids[5, 1] = 8          # out of range
        ids[6, 0] = -7         # out of range
        ids[9, 2] = -1
        s[9, 2] = 0.25         # inactive route carrying a score (debug flag)
        return Case(w, ids=ids, scores=s)
    if name == "dense":
        w = synth.Workload("dense", 96, 128, 128, 1, 1, "bf16", "uniform", seed=9)
        return Case(w, ids=np.zeros((96, 1), np.int32), scores=np.ones((96, 1), np.float32))
    if name == "one_token":
        w = synth.Workload("one", 1, 128, 128, 4, 2, "bf16", "uniform", seed=10)
        return Case(w)
    if name == "e1024":
        # the largest expert count: ids need all 10 bits the lane grouping compares
        w = synth.Workload("e1024", 256, 128, 128, 1024, 8, "bf16", "uniform", inactive_frac=0.1, seed=11)
        return Case(w)
    if name == "top_id_and_inactive":
        # E = 64: id 63 has every compared bit set, like -1; the grouping must still keep them apart,
        # and repeated ids inside one token count as separate routes
        w = synth.Workload("top", 128, 128, 128, 64, 6, "bf16", "uniform", seed=12)
        rng = np.random.default_rng(12)
        ids = rng.choice(np.array([63, 63, -1, 62, 0, 31], np.int32), size=(128, 6))
        s = rng.random((128, 6)).astype(np.float32)
        s[ids < 0] = 0.0
        return Case(w, ids=ids, scores=s)
    raise ValueError(name)


@pytest.mark.parametrize("name", ["tiny", "skewed", "bad_ids", "dense", "one_token", "e1024", "top_id_and_inactive"])
def test_routing_bit_exact(name):
    case = _routing_case(name)
    w = case.w
    res = run_gpu(case, training=True, backward=False, debug=True)
    layer, saved = res["layer"], res["saved"]
    from mixture_experts_routed_route_gb300 import abi
    E, T, K = w.E, case.T, w.K
    rt = omoe.route(case.ids, E)

    def field(f, dtype, n):
        return layer.saved_field(saved, f, dtype, (n,)).cpu().numpy()

    hdr = field(abi.MOE_SAVED_HEADER, torch.int32, 16)
    assert hdr[0] == T
    assert hdr[2] == rt.poffsets[E]
    assert hdr[3] == rt.num_active
    np.testing.assert_array_equal(field(abi.MOE_SAVED_COUNTS, torch.int32, E), rt.counts)
    np.testing.assert_array_equal(field(abi.MOE_SAVED_OFFSETS, torch.int32, E + 1), rt.offsets)
    np.testing.assert_array_equal(field(abi.MOE_SAVED_POFFSETS, torch.int32, E + 1), rt.poffsets)
    rows = int(rt.poffsets[E])
    np.testing.assert_array_equal(field(abi.MOE_SAVED_PERM, torch.int32, rows), rt.perm)
    np.testing.assert_array_equal(field(abi.MOE_SAVED_INV, torch.int32, T * K), rt.inv)
    sc = field(abi.MOE_SAVED_SCORES, torch.float32, T * K)
    np.testing.assert_array_equal(sc, np.where(rt.inv >= 0, case.scores.reshape(-1), 0.0).astype(np.float32))
    # row blocks: each expert's padded rows cut into <=128-row blocks, in order
    blocks = field(abi.MOE_SAVED_BLOCKS, torch.int32, 4 * int(hdr[1])).reshape(-1, 4)
    exp = []
    for e in range(E):
        pc = int(rt.poffsets[e + 1] - rt.poffsets[e])
        for b in range((pc + 127) // 128):
            exp.append([e, int(rt.poffsets[e]) + 128 * b, min(128, pc - 128 * b), 0])
    # pairs of consecutive blocks of one expert (the last alone when odd), in
    # word 3 of the first entries
    pairs = []
    b0 = 0
    for e in range(E):
        nbe = (int(rt.poffsets[e + 1] - rt.poffsets[e]) + 127) // 128
        pairs += [((b0 + j) << 1) | int(j + 1 < nbe) for j in range(0, nbe, 2)]
        b0 += nbe
    assert hdr[4] == len(pairs)
    for i, d in enumerate(pairs):
        exp[i][3] = d
    np.testing.assert_array_equal(blocks, np.array(exp, dtype=np.int32).reshape(-1, 4))
    # first block of each expert, and the block of every 32-row group
    nb = np.array([(int(rt.poffsets[e + 1] - rt.poffsets[e]) + 127) // 128 for e in range(E)])
    np.testing.assert_array_equal(field(abi.MOE_SAVED_BSTART, torch.int32, E + 1),
                                  np.concatenate([[0], np.cumsum(nb)]))
    rb = field(abi.MOE_SAVED_ROWBLOCK, torch.int32, rows // 32)
    for b, (_, r0, n, _) in enumerate(exp):
        assert np.all(rb[r0 // 32:(r0 + n) // 32] == b)
    # error word: bad IDs flagged; an inactive route with a score flagged in debug mode
    bits = res["err_bits"]
    assert bool(bits & abi.MOE_DEV_ERR_BAD_ID) == bool(rt.bad_ids.any())
    inactive_scored = np.any((case.ids.reshape(-1) == -1) & (case.scores.reshape(-1) != 0))
    assert bool(bits & abi.MOE_DEV_ERR_INACTIVE_SCORE) == bool(inactive_scored)
    assert not bits & abi.MOE_DEV_ERR_TIMEOUT
