"""Oracle of the activation-slot planner.  TEST INFRASTRUCTURE ONLY (see
``oracle/__init__``).

"Dist-MoE: Speed-of-light distributed Mixture-of-Experts kernels", section 04
"Activation Packing and Dynamic Recompute": several layers stack their saved
state in one slot buffer, each at the slot's running byte cursor (offsets
rounded to 128 bytes).  Before a layer keeps its full state, the planner
adds its full-state bytes to what the slot already holds, plus one input's
bytes for every layer still to come (their inputs must stay available for
replay); if the sum exceeds the slot's capacity the layer keeps only its
input and the backward replays it.  The page takes the maximum over EP
ranks of the first two terms; with one GPU there is one rank.  Backwards run
in reverse order and put the cursor back where their forward found it.

Reading where the page is silent: a layer that cannot keep even its input
(cursor + input + reserve > capacity) is an error rather than a silent
overflow.

Parity status: pinned by ``tests/test_slot_plan_cpu.py`` against the worked
example the page prints (``tests/golden/slot_plan_worked_example.json``) and
by brute-force properties.
"""

FULL = "full"
INPUT = "input"


def align128(n):
    """The page's align128(n) = ceil(n / 128) * 128."""
    return -(-int(n) // 128) * 128


def decide(cursor, full_bytes, input_bytes, remaining_layers, capacity):
    """(decision, bytes the layer takes, the test's left-hand side) for one
    layer whose state would start at `cursor`."""
    full, inp = align128(full_bytes), align128(input_bytes)
    reserve = remaining_layers * inp
    need_full = cursor + full + reserve
    if need_full <= capacity:
        return FULL, full, need_full
    if cursor + inp + reserve <= capacity:
        return INPUT, inp, need_full
    raise MemoryError("the slot cannot hold every remaining layer's input")


def plan_stack(layers, capacity):
    """Forward pass over a stack: `layers` is a list of (full_bytes,
    input_bytes); layer i has len(layers) - 1 - i layers after it, each
    reserved at that layer's input bytes (the page's remaining_layers x
    saved_input_bytes, with every layer's input the same size).

    Returns a list of dicts: offset, decision, bytes taken, and `need` (the
    full-state test's left-hand side)."""
    out = []
    cursor = 0
    n = len(layers)
    for i, (f, inp) in enumerate(layers):
        d, take, need = decide(cursor, f, inp, n - 1 - i, capacity)
        out.append({"offset": cursor, "decision": d, "bytes": take, "need": need})
        cursor += take
    return out
