"""Static rules of the CUDA sources (no GPU): every loop that polls for
another agent's progress gives up after a bounded time, and nothing in
device code traps, so a stuck wait or a bad input ends in an error bit and
a usable context rather than a lost GPU."""

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mixture_experts_routed_route_gb300", "csrc")


def _sources():
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh")):
            text = open(os.path.join(CSRC, name)).read()
            # comments may describe what the code avoids; only code counts
            text = re.sub(r"//[^\n]*", "", text)
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            yield name, text


def test_no_trap_or_device_assert():
    for name, text in _sources():
        assert "__trap" not in text, name
        assert not re.search(r"\btrap\s*;", text), name
        assert not re.search(r"(?<![\w.])assert\s*\(", text), name
        assert "__brkpt" not in text, name


def test_every_polling_loop_is_bounded():
    """Each while/for(;;) loop is either a do { } while (0) macro or polls with
    a clock64() deadline inside its body."""
    found = 0
    for name, text in _sources():
        for m in re.finditer(r"\bwhile\s*\(([^()]*(?:\([^()]*\)[^()]*)*)\)|\bfor\s*\(\s*;\s*;\s*\)", text):
            if m.group(0).startswith("while") and m.group(1).strip() == "0":
                continue
            if m.group(0).startswith("while"):
                # a do { } while (cond) tail has no body after it
                after = text[m.end():m.end() + 2].strip()
                if after.startswith(";"):
                    raise AssertionError(f"{name}: do/while loop without a deadline: {m.group(0)}")
            body_start = text.find("{", m.end())
            depth, i = 0, body_start
            while True:
                if text[i] == "{":
                    depth += 1
                elif text[i] == "}":
                    depth -= 1
                    if depth == 0:
                        break
                i += 1
            body = text[body_start:i]
            assert "clock64()" in body and ("return" in body or "break" in body), \
                f"{name}: polling loop without a deadline: {m.group(0)}"
            found += 1
    assert found >= 2      # the mbarrier wait and the drain wait


def test_kernel_setup_is_per_device():
    """Kernel attributes (the dynamic shared-memory opt-in) belong to the
    context of the current device: their one-time set-up is kept per device
    and under a lock, never in a process-wide flag."""
    for name, text in _sources():
        assert not re.search(r"static\s+bool\s+\w*configured", text), name
        if "cudaFuncSetAttribute" in text:
            assert "PerDeviceOnce" in text or "g_setup" in text, name
