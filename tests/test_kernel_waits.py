"""Every spin-wait in the CUDA sources gives up after a time limit.

A wait on an mbarrier phase, a ready word or a drain that never ends would hang the
GPU, so each `while` loop of the kernels must either read the global timer (and so
be bounded by a limit) or be one of the finite index loops listed below.  Checked on
the source text, without a GPU.
"""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "fp8_block_scaled_gb300", "csrc")

# loops whose trip count is bounded by their indices, not by another agent
FINITE = (
    "hi - lo > 1",        # binary search over group prefixes
    "pos < sk_end",       # walk over this pair's stream-K run
)


def _loops(text):
    """(line number, condition, body) of every while loop, body up to its closing brace."""
    for m in re.finditer(r"\bwhile\s*\(", text):
        i, depth = m.end(), 1
        while depth:
            depth += {"(": 1, ")": -1}.get(text[i], 0)
            i += 1
        cond = text[m.end():i - 1]
        body = ""
        j = i
        while j < len(text) and text[j] in " \t\n":
            j += 1
        if j < len(text) and text[j] == "{":
            k, depth = j + 1, 1
            while depth:
                depth += {"{": 1, "}": -1}.get(text[k], 0)
                k += 1
            body = text[j:k]
        yield text.count("\n", 0, m.start()) + 1, cond, body


def test_every_wait_loop_is_bounded():
    checked = 0
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh")):
            continue
        text = open(os.path.join(CSRC, name)).read()
        for line, cond, body in _loops(text):
            checked += 1
            if any(f in cond for f in FINITE):
                continue
            assert "global_timer_ns" in cond + body, f"{name}:{line}: unbounded wait `{cond}`"
    assert checked >= 8


def test_try_wait_is_only_polled_inside_bounded_loops_or_helpers():
    # mbar_try_wait is a single poll; outside the wait helpers it may appear only
    # in a loop condition that also reads the timer
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh")):
            continue
        for n, ln in enumerate(open(os.path.join(CSRC, name)), 1):
            if "mbar_try_wait(" not in ln or "bool mbar_try_wait" in ln:
                continue
            s = ln.strip()
            ok = (s.startswith("if (mbar_try_wait(") and "return true" in s) or \
                 ("while" in s and ("global_timer_ns" in s or s.endswith("&&")))
            assert ok, f"{name}:{n}: {s}"
