"""Plain fp64 CPU oracle for the dropless routed-expert MoE layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the
CUDA library; the two meet only through the seeded input generator, which
holds none of the method's arithmetic.

Modules
-------
formats    -- BF16 / FP32 / E4M3 / E8M0 rounding and the MX block quantisers.
moe        -- routing (counting sort), forward, backward, and the brute-force
              per-token forward used to pin the routed forward.
sample     -- bounded samples of a workload (routes of chosen experts).
post_norm  -- the post-expert RMSNorm and its backward.
slot_plan  -- the activation-slot save-or-replay decision rule.

Parity status: every function here is pinned, by ``tests/test_oracle_pins.py``
(closed forms, library routines, brute force, finite differences) or, for
the slot planner, by ``tests/test_slot_plan_cpu.py`` (the worked example the
page prints and brute-force properties).
"""

from . import formats, moe  # noqa: F401
