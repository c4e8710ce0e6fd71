"""The launchers' instance choice (csrc/dispatch.h), on the CPU.

The rules are host arithmetic over the problem size and the SM count; a small driver
(tests/dispatch_driver.cpp) built with the host compiler prints the choice for a table
of problems.  The expected choices are the measured ones on a 152-SM GB300 (the
timings behind each rule are stated beside it in dispatch.h), and the stream-K
schedule is checked against its definition: split only when whole tiles would leave
more than three quarters of the units idle and every unit gets at least 12 k-blocks.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PAIR256, SINGLE256, SINGLE128, SINGLE64 = 0, 1, 2, 3


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("dispatch") / "dispatch_driver")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "cute_layouts_mma_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "dispatch_driver.cpp"), "-o", exe], check=True)
    return exe


def choose(driver, problems, sms=152):
    args = [str(sms)] + [str(x) for p in problems for x in p]
    out = subprocess.run([driver, *args], check=True, capture_output=True, text=True).stdout.split("\n")
    return [tuple(int(v) for v in line.split()) for line in out if line.strip()]


# (M, N, K, k-coordinates per stage) -> (dense instance, stream-K split, block-scaled pair)
CASES = [
    ((4096, 4096, 4096, 64), (PAIR256, 0, 1)),      # the FP16 headline: 256 pair tiles
    ((8192, 8192, 1024, 64), (PAIR256, 0, 1)),
    ((4096, 4096, 1024, 64), (PAIR256, 0, 1)),      # 256 pair tiles: pairs (24.0 against 26.5 us)
    ((256, 256, 256, 64), (SINGLE64, 0, 0)),        # latency-bound: 128 x 64 tiles
    ((1024, 1024, 1024, 64), (SINGLE64, 0, 0)),
    ((2048, 2048, 1024, 64), (SINGLE256, 0, 1)),    # 64 pair tiles: single CTAs, whole tiles
    ((512, 8192, 2048, 64), (SINGLE256, 0, 1)),    # 64 pair tiles: dense single CTAs, block-scaled pairs
    ((1024, 1024, 4096, 64), (SINGLE128, 0, 0)),    # 256-wide tiles would split: 128-wide, whole
    ((256, 2048, 8192, 64), (SINGLE128, 1, 0)),     # 128-wide with stream-K
    ((128, 2560, 16384, 64), (SINGLE128, 1, 0)),
    ((128, 4096, 4096, 64), (SINGLE256, 0, 0)),     # shares too short to split: whole tiles
    ((128, 16384, 8192, 128), (SINGLE256, 0, 0)),   # the MXFP8 skinny shape; block-scaled: single
    ((1024, 2560, 8192, 128), (SINGLE256, 0, 1)),   # 40 pair tiles: block-scaled pairs
    ((512, 4096, 8192, 128), (SINGLE256, 0, 0)),    # 32 pair tiles: block-scaled single CTAs
    ((8192, 8192, 8192, 128), (PAIR256, 0, 1)),
]


def test_measured_choices(driver):
    got = choose(driver, [c[0] for c in CASES])
    for (problem, want), g in zip(CASES, got):
        assert g == want, (problem, g, want)


def _schedule_splits(tiles, nkb, units):
    """The stream-K rule restated: split the last round's tiles when more than 3/4 of
    the units would idle and the split tiles give every unit at least 12 k-blocks."""
    rounds = -(-tiles // units)
    idle = 1 - tiles / (rounds * units)
    split = tiles % units
    return idle > 0.75 and split * nkb >= 12 * units


@pytest.mark.parametrize("sms", [152, 148, 132])
def test_stream_k_rule_on_single_128(driver, sms):
    # problems the single-CTA 128 x 128 instance takes; the driver's split flag must
    # follow the rule for that instance's own tiles
    problems = [(M, N, K, 64) for M in (128, 256, 640) for N in (1024, 2560, 8192) for K in (2048, 16384, 65536)]
    for (M, N, K, kpb), (inst, split, _) in zip(problems, choose(driver, problems, sms)):
        if inst != SINGLE128:
            continue
        tiles = -(-M // 128) * -(-N // 128)
        assert split == int(_schedule_splits(tiles, -(-K // kpb), sms)), (M, N, K, sms)


def test_pairs_need_filled_sm_pairs(driver):
    # dense pairs exactly when the 256 x 256 tiles fill every SM pair (M > 128);
    # block-scaled pairs from half of them
    problems = [(M, N, 4096, 64) for M in (128, 256, 1024, 2048, 4096) for N in (256, 2048, 4864, 9728)]
    for (M, N, _, _), (inst, _, bs_pair) in zip(problems, choose(driver, problems)):
        pair_tiles = -(-M // 256) * -(-N // 256)
        assert (inst == PAIR256) == (M > 128 and pair_tiles >= 76), (M, N)
        assert bs_pair == int(M > 128 and 2 * pair_tiles >= 76), (M, N)
