"""Bounded samples of a full-size workload for the oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

A sample keeps every token but only the routes to a chosen set of experts
(the others become inactive, ID -1).  Routing is stable by flat route index,
so each chosen expert keeps exactly the rows, in the same order and with the
same 32-row blocks, that it has in the full problem: its h1/h2/h3 rows, its
dh3/dh1/dxr rows and its weight gradients equal those of the full problem,
and a token whose K experts are all chosen gets its full out and dX.
"""

import numpy as np

from . import moe


def restrict_routes(ids, experts):
    """IDs of a sample: expert experts[i] becomes i, every other route -1."""
    ids = np.asarray(ids)
    remap = np.full(max(int(ids.max(initial=0)) + 1, 1), -1, dtype=np.int64)
    for i, e in enumerate(experts):
        if e < remap.size:
            remap[e] = i
    out = np.where(ids >= 0, remap[np.clip(ids, 0, remap.size - 1)], -1)
    return out.astype(np.int64)


def useful_flops(ids, D, F, backward):
    """6 R D F forward, twice that again for backward (R = active routes)."""
    R = int(np.sum(np.asarray(ids) >= 0))
    return 6.0 * R * D * F * (3.0 if backward else 1.0)


def run(x, ids, scores, w13_sub, w2_sub, experts, precision, dY=None, **variant):
    """Oracle forward (and backward when dY is given) of the sample;
    ``variant`` passes swiglu_limit / weight_blocks to the forward."""
    sub_ids = restrict_routes(ids, experts)
    st = moe.forward(x, sub_ids, scores, w13_sub, w2_sub, precision, **variant)
    res = {"state": st, "ids": sub_ids, "out": st["out"]}
    if dY is not None:
        res["grads"] = moe.backward(st, dY, w13_sub, w2_sub)
    return res
