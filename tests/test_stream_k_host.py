"""The stream-K partition of csrc/stream_k.cuh (shared by the FP32 SIMT and
CTA-pair kernels), compiled for the host and checked against its
definition: worker c owns units [c*U/G, (c+1)*U/G) of the tail's units laid
end to end; a tile's workers are exactly those whose ranges meet it; its
finisher is the one whose share ends latest within its own range (the first
on a tie); and the finishers' waits can never form a cycle, so every wait
ends once the workers run (they are all resident)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "roofline_driven_optimisation_gb300", "csrc")
OUT = os.path.join(ROOT, "roofline_driven_optimisation_gb300", "_build", "sk_check")


@pytest.fixture(scope="module")
def sk():
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "sk_check.cpp"), "-o", OUT], check=True)

    def ask(tiles, upt, G):
        r = subprocess.run([OUT], input=f"{tiles} {upt} {G}\n", capture_output=True, text=True,
                           check=True)
        lines = r.stdout.split("\n")
        parts = [tuple(int(x) for x in l.split()) for l in lines[:tiles]]
        share = int(lines[tiles].split()[1])
        return parts, share
    return ask


def begin(c, U, G):
    return c * U // G


# (tail tiles, K-steps per tile, workers): the FP32 tail of 4096^3 (56 tiles of
# 256 slices on 152 CTAs) and of other shapes, the pair kernel's tails
# (76 pairs), workers fewer than, equal to and above the tiles
CASES = [(56, 256, 152), (128, 256, 152), (9, 64, 36), (1, 16, 1), (28, 64, 76), (52, 12, 76),
         (6, 64, 48), (16, 9, 18), (151, 16, 152), (3, 100, 3), (7, 1000, 152), (1, 4096, 152)]


@pytest.mark.parametrize("tiles,upt,G", CASES)
def test_partition_matches_its_definition(sk, tiles, upt, G):
    parts, share = sk(tiles, upt, G)
    U = tiles * upt
    covered = [0] * tiles
    for t, (c0, c1, fin) in enumerate(parts):
        T0, T1 = t * upt, (t + 1) * upt
        meet = [c for c in range(G) if begin(c + 1, U, G) > T0 and begin(c, U, G) < T1]
        assert (c0, c1) == (meet[0], meet[-1]), t
        assert meet == list(range(c0, c1 + 1))
        ends = {c: min(begin(c + 1, U, G), T1) - begin(c, U, G) for c in meet}
        best = max(ends.values())
        assert fin == min(c for c in meet if ends[c] == best), t
        for c in meet:
            covered[t] += min(begin(c + 1, U, G), T1) - max(begin(c, U, G), T0)
    assert covered == [upt] * tiles          # every unit of every tile, once
    assert share == max(c1 - c0 + 1 for c0, c1, _ in parts)


@pytest.mark.parametrize("tiles,upt,G", [c for c in CASES if c[2] >= c[0]])
def test_ranges_touch_at_most_two_tiles_and_waits_are_acyclic(sk, tiles, upt, G):
    # with at least as many workers as tiles no range is longer than a tile:
    # a worker has at most two pieces (the kernels' kSkMaxSeg), the first
    # ending its range in one tile and the second starting in the next
    parts, _ = sk(tiles, upt, G)
    U = tiles * upt
    pieces = {c: [] for c in range(G)}
    for t, (c0, c1, fin) in enumerate(parts):
        for c in range(c0, c1 + 1):
            pieces[c].append(t)
    assert all(len(v) <= 2 for v in pieces.values())
    assert all(len(v) < 2 or v[1] == v[0] + 1 for v in pieces.values())
    # a worker's pieces run in order; a finisher's piece waits for the other
    # pieces of its tile; no cycle may run through these edges
    node = lambda c, t: (c, pieces[c].index(t))
    deps = {}
    for t, (c0, c1, fin) in enumerate(parts):
        for c in range(c0, c1 + 1):
            d = deps.setdefault(node(c, t), [])
            if node(c, t)[1] == 1:
                d.append((c, 0))
            if c == fin:
                d.extend(node(w, t) for w in range(c0, c1 + 1) if w != c)
    state = {}

    def visit(x):
        state[x] = 1
        for y in deps.get(x, []):
            assert state.get(y) != 1, f"wait cycle through {x} and {y}"
            if y not in state:
                visit(y)
        state[x] = 2
    for x in list(deps):
        if x not in state:
            visit(x)
