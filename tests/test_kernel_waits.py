"""Source checks of the CUDA kernels that need no GPU: every spin-wait gives up
after a time limit, and every tiled TMA copy starts on a 16-byte boundary.

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


def _call_args(text, start):
    """Top-level comma-separated arguments of the call whose '(' is at text[start]."""
    args, depth, cur = [], 0, ""
    for ch in text[start + 1:]:
        if ch in "([{":
            depth += 1
        elif ch in ")]}":
            if depth == 0:
                args.append(cur.strip())
                return args
            depth -= 1
        if ch == "," and depth == 0:
            args.append(cur.strip())
            cur = ""
        else:
            cur += ch
    raise AssertionError("unbalanced call")


def test_tma_inner_coordinate_is_16_byte_aligned():
    # A tiled TMA copy must start its innermost coordinate on a 16-byte boundary; with
    # byte-sized elements every call passes 0 or a whole number of 128-byte K blocks.
    allowed = {"0", "kb * kBK"}
    calls = 0
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh")):
            continue
        text = open(os.path.join(CSRC, name)).read()
        for m in re.finditer(r"\b(tma_load_[23]d(?:_pair)?|tma_prefetch_[23]d)\s*\(", text):
            line = text.count("\n", 0, m.start()) + 1
            before = text[text.rfind("\n", 0, m.start()):m.start()]
            if "__device__" in before or "inline" in before or "//" in before:
                continue  # the definition, or a mention in a comment
            args = _call_args(text, m.end() - 1)
            x = args[1] if m.group(1).startswith("tma_prefetch") else args[2]
            calls += 1
            assert x in allowed, f"{name}:{line}: inner coordinate `{x}`"
    assert calls >= 6
