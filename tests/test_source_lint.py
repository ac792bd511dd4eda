"""Static checks of the CUDA sources that need no GPU.

A warp-synchronous intrinsic with a full mask must be executed by every lane
named in the mask; one placed behind a short-circuit operator (&&, ||, ?:)
is skipped by some lanes and the others wait for them forever."""

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "combine_get_layout_gb300", "csrc")

SYNC = re.compile(r"__(match_any|match_all|shfl\w*|ballot|any|all|reduce_\w+)_sync\s*\(")


def _statements(text):
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return text.split(";")


def test_no_warp_sync_intrinsic_behind_short_circuit():
    bad = []
    for fn in sorted(os.listdir(CSRC)):
        if not fn.endswith((".cu", ".cuh")):
            continue
        for st in _statements(open(os.path.join(CSRC, fn)).read()):
            m = SYNC.search(st)
            if not m:
                continue
            before = st[: m.start()]
            # the statement part after the last '{' or ')' that closes a
            # control header is the expression holding the call
            expr = before.split("{")[-1]
            if re.search(r"&&|\|\||\?", expr):
                bad.append((fn, " ".join(st.split())[:160]))
    assert not bad, bad


def test_lint_catches_the_pattern():
    st = "if (e >= 0 && __popc(__match_any_sync(0xffffffffu, key)) > 1) x = 1"
    m = SYNC.search(st)
    assert m and re.search(r"&&|\|\||\?", st[: m.start()].split("{")[-1])
