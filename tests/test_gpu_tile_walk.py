"""The grouped GEMMs' persistent CTAs take every grid-th tile and advance
its coordinates (block and slice; expert, m and n for the weight gradient)
with carries instead of dividing the tile index.  Small cases have fewer
tiles than SMs, so each CTA gets one tile; capping the grid
(moe_ctx_set_max_ctas) makes every CTA walk many tiles across slice, block
and expert boundaries.  Each output tile is computed by one CTA with the
same instruction sequence, so a capped run must equal the default run bit
for bit, forward and backward; the default run is checked against the
oracle by the forward and backward parity tests.
"""

import numpy as np
import pytest

from mixture_experts_routed_route_gb300 import abi, synth

from moe_cases import TOL, Case, rel_err, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

KEYS = ("out", "dx", "dW13", "dW2", "dp")


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_capped_grids_are_bit_exact(precision):
    # D=512, F=384, E=12: W13 WGRAD has 6 x 4 tiles per expert, W2 WGRAD
    # 4 x 3; W2 forward and W13 DGRAD two 256-wide slices; W13 forward three
    # gate/up slices.  Steps 3, 7 and 13 carry n into m and m into e.
    w = synth.Workload(f"walk_{precision}", 300, 512, 384, 12, 3, precision, "zipf", inactive_frac=0.05,
                       zipf_s=1.2, seed=51)
    case = Case(w)
    ref = run_gpu(case)
    assert ref["err_bits"] == 0
    assert rel_err(ref["out"], run_oracle(case, backward=False)["out"]) <= TOL[precision]
    for cap in (1, 3, 7, 13):
        g = run_gpu(case, max_ctas=cap)
        assert g["err_bits"] == 0
        for k in KEYS:
            np.testing.assert_array_equal(g[k], ref[k], err_msg=f"{k}, grid capped at {cap}")


def test_max_ctas_rejects_negative():
    from mixture_experts_routed_route_gb300.layer import MoELayer
    layer = MoELayer(64, 256, 256, 4, 2, "bf16", training=False)
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_ctx_set_max_ctas(layer.ctx, -1)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    abi.moe_ctx_set_max_ctas(layer.ctx, 0)
    layer.close()
