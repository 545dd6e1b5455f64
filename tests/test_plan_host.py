"""Launch planning on the CPU: the wave models of csrc/plan.h, compiled with
g++ into a small query program, checked against choices measured on GB300
(152 SMs; 76 clusters of four resident FP32 CTAs per GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "roofline_driven_optimisation_gb300", "csrc")
OUT = os.path.join(ROOT, "roofline_driven_optimisation_gb300", "_build", "plan_check")


@pytest.fixture(scope="module")
def plan():
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "plan_check.cpp"), "-o", OUT], check=True)

    def ask(*queries):
        text = "".join(" ".join(str(x) for x in q) + "\n" for q in queries)
        r = subprocess.run([OUT], input=text, capture_output=True, text=True, check=True)
        return r.stdout.split("\n")[:len(queries)]
    return ask


SMS = 152


def tc(plan, M, N, allowed=1):
    return tuple(int(x) for x in plan(("tc", M, N, SMS, allowed))[0].split())


def test_tensor_core_config_measured_choices(plan):
    # square and LLaMA-7B prefill shapes: 256-wide CTA pairs were fastest of
    # every configuration timed (within 1 %)
    for M, N in ((4096, 4096), (8192, 8192), (2048, 12288), (2048, 4096), (2048, 11008),
                 (2048, 32000), (1024, 4096), (3072, 4096), (4096, 2048)):
        assert tc(plan, M, N) == (2, 256), (M, N)
    # a small M: 128-wide pairs (22.5 us for 256 x 4096 x 4096, the same as
    # 256-wide pairs whose every tile is halved; the tie keeps 128)
    assert tc(plan, 256, 4096) == (2, 128)


def test_tensor_core_config_counts_the_halved_last_wave(plan):
    # shapes where 256-wide pairs with a halved last wave beat the single-CTA
    # 192-wide tiles or 128-wide pairs the model picked without the split
    # (GB300, K = 4096: 5-14 % faster)
    for M, N, without in ((512, 11008, (1, 192)), (1024, 11008, (2, 128)),
                          (2048, 3072, (1, 192)), (1536, 4096, (1, 192))):
        assert tc(plan, M, N) == (2, 256), (M, N)
        assert tc(plan, M, N, allowed=0) == without, (M, N)


def test_pair_stream_k_pairs(plan):
    # every pair streams at least 8 K-steps, and no range may span three
    # tiles (at least as many pairs as tail tiles)
    ask = lambda rem, k: int(plan(("tcsk", rem, k, 76))[0])
    assert ask(28, 64) == 76       # bf16 4096^3: 28 tail tiles, 64 K-steps each
    assert ask(6, 64) == 48        # 6 tiles x 64 / 8
    assert ask(16, 9) == 18
    assert ask(16, 4) == 0         # fewer than 8 K-steps a tile
    assert ask(100, 8) == 0        # 100 tiles, at most 76 pairs: a range would span 3 tiles
    assert ask(0, 64) == 0


def test_pair_tail_choice(plan):
    # measured on GB300: half-width tiles beat whole tiles, and stream-K (its
    # fix-up on the critical path) loses to both, so it is never chosen
    ask = lambda rem, half, sk: int(plan(("tctail", rem, 76, half, sk))[0])
    assert ask(28, 1, 76) == 1     # bf16 4096^3: half-width
    assert ask(52, 0, 76) == 0     # o-proj 2048 x 4096: halves do not fit
    assert ask(28, 0, 76) == 0     # FP8 (no half-width tiles)
    assert ask(12, 1, 76) == 1     # lm head 2048 x 32000
    assert ask(0, 1, 76) == 0


def test_single_cta_tile_width(plan):
    # single-CTA tiles timed on GB300 at K = 4096 (256 / 192 / 128 wide):
    # 512 x 11008: 62.3 / 51.2 / 52.4 us; 1024 x 4096: 33.0 / 45.2 / 34.8 us;
    # 4096 x 4096: 100.8 / 98.3 / 98.8 us (the model's 128 is within 0.5 %)
    assert plan(("bn", 512, 11008, SMS), ("bn", 1024, 4096, SMS),
                ("bn", 4096, 4096, SMS)) == ["192", "256", "128"]


def simt(plan, M, N, K, clusters=76, allowed=1):
    tiles = -(-M // 128) * -(-N // 128)
    return plan(("simt", tiles, -(-K // 16), SMS, clusters, 4, 10, allowed))[0] == "1"


def test_fp32_split_last_wave_choices(plan):
    # split on GB300 and faster there (single launch -> split)
    assert simt(plan, 4096, 4096, 4096)      # 2.377 -> 2.351 ms
    assert simt(plan, 4096, 4352, 4096)      # 2.704 -> 2.444 ms
    assert simt(plan, 2048, 2048, 4096)      # 0.709 -> 0.611 ms
    assert simt(plan, 1024, 1024, 4096)      # 0.375 -> 0.186 ms
    assert simt(plan, 2560, 2048, 1024)      # 0.275 -> 0.205 ms
    # left whole: the partial wave already runs one CTA per SM, or there is none
    assert not simt(plan, 4096, 3584, 4096)  # 896 tiles: 288 past two waves
    assert not simt(plan, 8192, 8192, 4096)  # 144 past 13 waves
    assert not simt(plan, 4864, 4096, 4096)  # 1216 tiles: four whole waves
    # too little K for four ranks of ten K-slices, or splitting forbidden
    assert not simt(plan, 1024, 1024, 624)
    assert simt(plan, 1024, 1024, 640)
    assert not simt(plan, 4096, 4096, 4096, allowed=0)
    # fewer resident clusters: 448 quarter-tiles need two full rounds
    assert not simt(plan, 4096, 4096, 4096, clusters=72)


def test_decode_cluster_split(plan):
    # LLaMA-7B decode: qkv, o, gate/up, down, lm column slabs of 128 (K = 4096
    # in 64 stages, down 11008 in 172): the largest power of two whose grid
    # fits two CTAs per SM
    got = plan(("cluster", 96, 64, SMS, 0, 8), ("cluster", 32, 64, SMS, 0, 8),
               ("cluster", 86, 64, SMS, 0, 8), ("cluster", 32, 172, SMS, 0, 8),
               ("cluster", 250, 64, SMS, 0, 8))
    assert got == ["2", "8", "2", "8", "1"]
    # a forced split, still clamped to the K units there are
    assert plan(("cluster", 250, 64, SMS, 4, 8), ("cluster", 32, 3, SMS, 0, 8),
                ("cluster", 32, 3, SMS, 8, 8)) == ["4", "2", "2"]


def simtopt(plan, tn, M, N, K, c2, c4, allowed=1):
    bn = 16 * tn
    tiles = -(-M // 128) * -(-N // bn)
    min_k = 10 if tn == 8 else 16   # two rounds of the 5- or 8-stage ring
    t, split = plan(("simtopt", tn, tiles, -(-K // 16), SMS, c2, c4, min_k, allowed))[0].split()
    return float(t), int(split)


def test_fp32_wide_tile_model(plan):
    # 4096^3 with 128 x 256 tiles: 512 tiles = 3 waves of 152 + 56; the 56
    # tiles' 56 x 256 K-slices spread over 152 CTAs (stream-K): 56/152 of a
    # wave plus 0.02 for the partial sums' exchange, against a whole fourth
    # round
    t, split = simtopt(plan, 16, 4096, 4096, 4096, 0, 0)
    assert split == 0
    assert t == pytest.approx(2 / 1.075 * (3 + 56 / 152 + 0.02), rel=1e-3)
    # forbidden split: a whole fourth round
    assert simtopt(plan, 16, 4096, 4096, 4096, 0, 0, allowed=0) == \
        (pytest.approx(2 / 1.075 * 4, rel=1e-3), 1)
    # few slices: the CTAs get at least 16 K-slices each (1024^2 x 512: 32
    # tiles x 32 slices over 64 CTAs)
    assert simtopt(plan, 16, 1024, 1024, 512, 0, 0) == (pytest.approx(2 / 1.075 * (32 / 64 + 0.02), rel=1e-3), 0)
    # fewer than 16 K-slices a tile: no stream-K
    assert simtopt(plan, 16, 1024, 1024, 240, 0, 0)[1] == 1
    # whole waves only (608 tiles = 4 x 152): nothing to split
    assert simtopt(plan, 16, 4864, 4096, 4096, 0, 0) == (pytest.approx(2 / 1.075 * 4, rel=1e-3), 1)


def test_fp32_narrow_tile_model_matches_the_split_rule(plan):
    # the 128 x 128 option is the wave model of simt_split: 4096^3 splits
    t, split = simtopt(plan, 8, 4096, 4096, 4096, 0, 76)
    assert split == 4
    assert t == pytest.approx(2 * (3 + 0.25 + 0.25 * 0.53), rel=1e-3)
    assert simtopt(plan, 8, 8192, 8192, 4096, 0, 76)[1] == 1


def test_fp32_tile_choice(plan):
    # the dispatcher takes the wide tiles when their estimate is below 0.97 of
    # the narrow one; the choices the GB300 timings favour (narrow / wide,
    # ms): 4096^3 2.339 / 2.285, 8192^2 x 4096 9.356 / 8.816, 4096 x 3584 x
    # 4096 2.115 / 1.971 on the wide tiles; 2048^2 x 4096 0.602 / 0.662,
    # 2560 x 2048 x 1024 0.210 / 0.224 and 256^3 (4 narrow tiles, one CTA
    # per SM) on the narrow ones
    def wide(M, N, K):
        return simtopt(plan, 16, M, N, K, 0, 0)[0] < 0.97 * simtopt(plan, 8, M, N, K, 0, 76)[0]
    for M, N, K in ((4096, 4096, 4096), (8192, 8192, 4096), (4096, 3584, 4096)):
        assert wide(M, N, K), (M, N, K)
    for M, N, K in ((2560, 2048, 1024), (256, 256, 256)):
        assert not wide(M, N, K), (M, N, K)
