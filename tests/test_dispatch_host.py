"""The launchers' instance choice (csrc/dispatch.h), on the CPU.

The rules are host arithmetic over the problem size and the SM count; a small driver
(tests/dispatch_driver.cpp) built with the host compiler prints the choices for a table
of problems, with co-resident cluster counts modelled as a device of 8 equal GPCs.
The expected choices are the measured ones on a 152-SM GB300 (the timings behind each
rule are stated beside it in dispatch.h), and the rules are also checked against their
definitions: the cluster split (largest s <= 8 with at least 4 k-blocks per CTA, at
most one CTA per SM, every tile's cluster resident, only when whole tiles leave more
than half of the SMs idle), the stream-K rule of the fixed-scratch call (split only
when whole tiles would leave more than three quarters of the units idle and every unit
gets at least 12 k-blocks), and the raster group (largest group up to 16 whose panels
fit the L2 budget).
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


def resident(sms, s):
    """The driver's model: clusters of s CTAs co-resident on 8 GPCs of sms / 8 SMs."""
    return 8 * ((sms // 8) // s)


# (M, N, K, k-coordinates per stage) -> (gemm_f16 / bf16 / fp8 instance, its cluster split),
# measured on GB300 (FP16, no C, graph replay; before -> after the cluster split, us)
PLAN_CASES = [
    ((4096, 4096, 4096, 64), (PAIR256, 1)),       # the FP16 headline: 256 pair tiles
    ((8192, 8192, 1024, 64), (PAIR256, 1)),
    ((4096, 4096, 1024, 64), (PAIR256, 1)),       # 256 pair tiles: pairs (24.0 against 26.5 us)
    ((256, 256, 256, 64), (SINGLE64, 1)),         # latency-bound: 128 x 64 tiles
    ((1024, 1024, 1024, 64), (SINGLE64, 1)),      # 7.2 us; split in clusters 12.6 us
    ((2048, 2048, 1024, 64), (SINGLE256, 1)),     # 64 pair tiles, short K: single CTAs (9.4 against 9.8)
    ((512, 8192, 2048, 64), (PAIR256, 1)),        # 64 pair tiles, long K: 17.5 -> 15.7 on pairs
    ((2048, 2048, 4096, 64), (PAIR256, 1)),       # 27.2 -> 24.4 on pairs
    ((1024, 1024, 4096, 64), (SINGLE128, 2)),     # 20.3 -> 14.4; 12.6 on 128 x 128 tiles
    ((256, 2048, 8192, 64), (SINGLE128, 4)),      # 24.9 -> 16.5 -> 14.7
    ((128, 4096, 4096, 64), (SINGLE128, 4)),      # 26.8 -> 12.2 -> 11.0
    ((128, 8192, 8192, 64), (SINGLE128, 2)),      # 37.6 -> 30.3 -> 26.9
    ((128, 2560, 16384, 64), (SINGLE128, 6)),     # 34.2 -> 22.4
    ((500, 760, 16384, 64), (SINGLE128, 6)),      # 31.3 -> 22.2
    ((8192, 8192, 8192, 128), (PAIR256, 1)),
]

# (M, N, K, k-coordinates per stage) -> (fixed-scratch instance, stream-K split, block-scaled pair)
FIXED_SCRATCH_CASES = [
    ((4096, 4096, 4096, 64), (PAIR256, 0, 1)),
    ((256, 256, 256, 64), (SINGLE64, 0, 0)),
    ((1024, 1024, 1024, 64), (SINGLE64, 0, 0)),
    ((2048, 2048, 1024, 64), (SINGLE256, 0, 1)),    # 64 pair tiles: single CTAs, whole tiles
    ((512, 8192, 2048, 64), (PAIR256, 0, 1)),       # 64 pair tiles, long K: pairs
    ((1024, 1024, 4096, 64), (SINGLE128, 0, 0)),    # 256-wide tiles would split: 128-wide, whole
    ((256, 2048, 8192, 64), (SINGLE128, 1, 0)),     # 128-wide with stream-K
    ((128, 2560, 16384, 64), (SINGLE128, 1, 0)),
    ((128, 4096, 4096, 64), (SINGLE256, 0, 0)),     # shares too short to split: whole tiles
    ((128, 16384, 8192, 128), (SINGLE256, 0, 0)),   # the MXFP8 skinny shape; block-scaled: single
    ((1024, 2560, 8192, 128), (PAIR256, 0, 1)),     # 40 pair tiles, long K: pairs (dense and block-scaled)
    ((512, 4096, 8192, 128), (SINGLE256, 0, 0)),    # 32 pair tiles: block-scaled single CTAs
    ((8192, 8192, 8192, 128), (PAIR256, 0, 1)),
]


def test_measured_dense_plans(driver):
    got = choose(driver, [c[0] for c in PLAN_CASES])
    for (problem, want), g in zip(PLAN_CASES, got):
        assert (g[3], g[4]) == want, (problem, g, want)


def test_fixed_scratch_choices(driver):
    got = choose(driver, [c[0] for c in FIXED_SCRATCH_CASES])
    for (problem, want), g in zip(FIXED_SCRATCH_CASES, got):
        assert g[:3] == want, (problem, g, want)


def _split_rule(tiles, nkb, sms):
    """The cluster split restated."""
    if tiles > sms or 1 - tiles / sms <= 0.5:
        return 1
    best = 1
    for s in range(2, 9):
        if nkb < 4 * s or tiles * s > sms:
            break
        if tiles <= resident(sms, s):
            best = s
    return best


@pytest.mark.parametrize("sms", [152, 148, 132])
def test_cluster_split_rule(driver, sms):
    # the block-scaled single-CTA instance (128 x 128 tiles) takes the rule as it stands
    problems = [(M, N, K, 128) for M in (128, 256, 640) for N in (512, 2560, 8192) for K in (1024, 8192, 65536)]
    for (M, N, K, kpb), g in zip(problems, choose(driver, problems, sms)):
        tiles = -(-M // 128) * -(-N // 128)
        assert g[5] == _split_rule(tiles, -(-K // kpb), sms), (M, N, K, sms)
        s = g[5]
        assert 1 <= s <= 8 and (s == 1 or (tiles * s <= sms and -(-K // kpb) >= 4 * s))


def _schedule_splits(tiles, nkb, units):
    """The stream-K rule restated: split the last round's tiles when more than 3/4 of
    the units would idle and the split tiles give every unit at least 12 k-blocks."""
    rounds = -(-tiles // units)
    idle = 1 - tiles / (rounds * units)
    split = tiles % units
    return idle > 0.75 and split * nkb >= 12 * units


@pytest.mark.parametrize("sms", [152, 148, 132])
def test_stream_k_rule_on_single_128(driver, sms):
    # problems the fixed-scratch call gives the single-CTA 128 x 128 instance; its split
    # flag must follow the rule for that instance's own tiles
    problems = [(M, N, K, 64) for M in (128, 256, 640) for N in (1024, 2560, 8192) for K in (2048, 16384, 65536)]
    for (M, N, K, kpb), g in zip(problems, choose(driver, problems, sms)):
        if g[0] != SINGLE128:
            continue
        tiles = -(-M // 128) * -(-N // 128)
        assert g[1] == int(_schedule_splits(tiles, -(-K // kpb), sms)), (M, N, K, sms)


def test_pairs_need_filled_sm_pairs(driver):
    # dense pairs when the 256 x 256 tiles fill every SM pair (M > 128), or half of them
    # with K >= 2048; block-scaled pairs from half of them
    problems = [(M, N, K, 64) for M in (128, 256, 1024, 2048, 4096) for N in (256, 2048, 4864, 9728) for K in (1024, 4096)]
    for (M, N, K, _), g in zip(problems, choose(driver, problems)):
        pair_tiles = -(-M // 256) * -(-N // 256)
        dense = M > 128 and (pair_tiles >= 76 or (K >= 2048 and 2 * pair_tiles >= 76))
        assert (g[0] == PAIR256) == dense, (M, N, K)
        assert (g[3] == PAIR256) == dense, (M, N, K)
        assert g[2] == int(M > 128 and 2 * pair_tiles >= 76), (M, N, K)


def test_raster_group_fits_the_budget(driver):
    # 256 x 256 pair tiles, k-coordinates of 128 bytes: panels of 256 rows x K bytes
    budget = 64 << 20
    problems = [(M, N, K, 128) for M in (512, 4096, 8192, 32768) for N in (1024, 8192, 65536) for K in (1024, 8192, 65536)]
    for (M, N, K, kpb), g in zip(problems, choose(driver, problems)):
        num_m, num_n, units = -(-M // 256), -(-N // 256), 76
        panel = 256 * (-(-K // kpb)) * 128
        group = g[6]
        assert 1 <= group <= min(16, num_m), (M, N, K, group)

        def fits(gr):
            wave = min(units, gr * num_n)
            return gr * panel + (-(-wave // gr) + 1) * panel <= budget

        assert group == 1 or fits(group), (M, N, K, group)
        assert group == min(16, num_m) or not fits(group + 1) or group + 1 > 16, (M, N, K, group)
