"""GPU parity of the CUDA TN GEMM against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import cute_layouts_mma_gb300 as tg
from cute_layouts_mma_gb300 import inputs
import oracle

import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tg.lib()


# ------------------------------------------------------------------ FP16, fp32 accumulation

def test_fp16_int_256_bit_exact():
    prob = inputs.workload_problem("fp16_int_256")
    D = P.run_gpu(prob, accum=0)
    P.check(prob, D, mode="exact")


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (128, 256, 64), (130, 264, 72), (300, 520, 200),
                                   (257, 8, 1000), (64, 1000, 4096), (1000, 16, 520)])
def test_fp16_ragged_shapes_tolerance(M, N, K):
    prob = inputs.make_problem("f16", M, N, K, seed=M + N + K, dist="normal0.1", with_c=True)
    D = P.run_gpu(prob, accum=0)
    P.check(prob, D, mode="tol")


def test_fp16_integers_with_c_bit_exact():
    prob = inputs.make_problem("f16", 384, 520, 512, seed=7, dist="int2", with_c=True)
    P.check(prob, P.run_gpu(prob, accum=0), mode="exact")


def test_fp16_in_place_and_null_c():
    prob = inputs.make_problem("f16", 200, 264, 136, seed=8, dist="int2", with_c=True)
    dev = P.device()
    g = P.to_device(prob, dev)
    D = g["C"].clone()
    tg.gemm_f16(g["A"], g["B"], D, D, tg.GEMM_ACC_F32)  # D is C
    torch.cuda.synchronize()
    P.check(prob, D.cpu(), mode="exact")
    prob0 = dict(prob, C=None)
    D0 = P.run_gpu(prob0, accum=0)
    Dz = P.run_gpu(dict(prob, C=torch.zeros_like(prob["C"])), accum=0)
    assert torch.equal(D0.view(torch.int16), Dz.view(torch.int16))
    P.check(prob0, D0, mode="exact")


def test_fp16_guard_bands_untouched():
    prob = inputs.make_problem("f16", 130, 136, 64, seed=9, dist="int2", with_c=False)
    M, N = 130, 136
    pad = 4096
    dev = P.device()
    buf = torch.full((M * N + 2 * pad,), float("nan"), dtype=torch.float16, device=dev)
    D = buf[pad:pad + M * N].view(M, N)
    P.run_gpu(prob, accum=0, D=D)
    host = buf.cpu()
    assert torch.isnan(host[:pad]).all() and torch.isnan(host[pad + M * N:]).all()
    P.check(prob, D.cpu(), mode="exact")


def test_fp16_side_stream():
    prob = inputs.make_problem("f16", 256, 512, 256, seed=10, dist="int2", with_c=True)
    s = torch.cuda.Stream()
    D = P.run_gpu(prob, accum=0, stream=s)
    P.check(prob, D, mode="exact")


def test_fp16_4096_full_size_sampled_rows():
    prob = inputs.workload_problem("fp16_4096")
    D = P.run_gpu(prob, accum=0)
    rows = P.sample_rows(prob["M"], 32, seed=1)
    info = P.check(prob, D, rows=rows, mode="tol")
    # the stated bound, output rounding included, without the extra half ulp
    d16, d64 = P.oracle_result(prob, rows)
    assert float(np.max(np.abs(D[rows].double().numpy() - d64))) <= P.tolerance_f32acc(prob)
    # properties at every row: finite, and equal to the same launch repeated
    assert torch.isfinite(D.float()).all()
    D2 = P.run_gpu(prob, accum=0)
    assert torch.equal(D.view(torch.int16), D2.view(torch.int16))


# ------------------------------------------------------------------ FP16 accumulation

@pytest.mark.parametrize("M,N,K,rows", [(512, 768, 8192, None), (4096, 4096, 8192, 24)])
def test_fp16_pairs_long_k_whole_tiles(M, N, K, rows):
    # CTA pairs over whole tiles with more k-blocks than the 4096^3 workload
    prob = inputs.make_problem("f16", M, N, K, seed=K + M, dist="normal0.1", with_c=True)
    D = P.run_gpu(prob, accum=0)
    P.check(prob, D, rows=None if rows is None else P.sample_rows(M, rows, seed=7), mode="tol")


@pytest.mark.parametrize("M,N,K", [(256, 264, 32), (128, 520, 16), (300, 256, 8), (100, 136, 24),
                                   (1000, 1000, 32), (129, 8, 16)])
def test_fp16_narrow_k_integers_bit_exact(M, N, K):
    # K of at most 32 / 16 elements: 64- / 32-byte operand rows with the matching swizzle
    prob = inputs.make_problem("f16", M, N, K, seed=M + K, dist="int2", with_c=True)
    P.check(prob, P.run_gpu(prob, accum=0), mode="exact")


@pytest.mark.parametrize("M,N,K", [(513, 384, 32), (64, 256, 16), (2048, 2048, 24)])
def test_fp16_narrow_k_random_tolerance(M, N, K):
    prob = inputs.make_problem("f16", M, N, K, seed=M + N + K, dist="normal0.1", with_c=True)
    P.check(prob, P.run_gpu(prob, accum=0), mode="tol")


def test_fp16acc_integers_bit_exact():
    # every partial sum is an integer of magnitude <= 1024: exact in fp16
    prob = inputs.make_problem("f16", 256, 264, 256, seed=11, dist="int2", with_c=False)
    P.check(prob, P.run_gpu(prob, accum=1), mode="exact")


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (200, 136, 328)])
def test_fp16acc_frobenius(M, N, K):
    prob = inputs.make_problem("f16", M, N, K, seed=12, dist="uniform0.5", with_c=False)
    P.check(prob, P.run_gpu(prob, accum=1), mode="fro")


def test_fp16acc_8192x1024_full_size_sampled_rows():
    prob = inputs.workload_problem("fp16acc_8192x1024")
    D = P.run_gpu(prob, accum=1)
    rows = P.sample_rows(prob["M"], 48, seed=2)
    P.check(prob, D, rows=rows, mode="fro")
    assert torch.isfinite(D.float()).all()


# ------------------------------------------------------------------ NVFP4

@pytest.mark.parametrize("with_c", [False, True])
def test_nvfp4_integers_bit_exact(with_c):
    prob = inputs.make_problem("nvfp4", 256, 512, 512, seed=13, dist="int", with_c=with_c)
    P.check(prob, P.run_gpu(prob), mode="exact")


@pytest.mark.parametrize("with_c", [True, False])
@pytest.mark.parametrize("M,N,K", [(200, 264, 768), (129, 8, 256), (384, 1024, 2048), (520, 200, 512)])
def test_nvfp4_random_tolerance(M, N, K, with_c):
    # M > 128 without C runs the instance that holds half of each slice in registers
    prob = inputs.make_problem("nvfp4", M, N, K, seed=M + K, dist="codes", with_c=with_c)
    P.check(prob, P.run_gpu(prob), mode="tol")


def _one_hot_problem(kind, M, N, K, row, col, sfk):
    kblk = 16 if kind == "nvfp4" else 32
    if kind == "nvfp4":
        A = torch.full((M, K // 2), 0x22, dtype=torch.uint8)
        B = torch.full((N, K // 2), 0x22, dtype=torch.uint8)
        s1, s2 = 0x38, 0x40
    else:
        A = torch.full((M, K), 0x38, dtype=torch.uint8)
        B = torch.full((N, K), 0x38, dtype=torch.uint8)
        s1, s2 = 127, 128
    SFA = torch.full((M, K // kblk), s1, dtype=torch.uint8)
    SFB = torch.full((N, K // kblk), s1, dtype=torch.uint8)
    if row is not None:
        SFA[row, sfk] = s2
    if col is not None:
        SFB[col, sfk] = s2
    return {"kind": kind, "M": M, "N": N, "K": K, "A": A, "B": B, "SFA": SFA, "SFB": SFB, "C": None}


# 256 x 264: single-CTA instance; 640 x 3328 (39 tiles of 256 x 256 for 76 SM pairs):
# CTA-pair instance, whose CTAs each hold all 256 SFB rows of a tile
@pytest.mark.parametrize("kind", ["nvfp4", "mxfp8"])
@pytest.mark.parametrize("row,col,sfk", [(0, None, 0), (37, None, 5), (None, 200, 6),
                                         (127, 129, 15), (64, None, 2), (None, 31, 3), (300, 2900, 9)])
@pytest.mark.parametrize("M,N,K", [(256, 264, 1024), (640, 3328, 512)])
def test_one_hot_scale_probe(kind, row, col, sfk, M, N, K):
    """All data 1 and all scales 1 except one SFA row or SFB column block set to 2:
    only that row / column of D moves, by K_blk."""
    if row is not None and row >= M or col is not None and col >= N:
        pytest.skip("probe outside this shape")
    prob = _one_hot_problem(kind, M, N, K, row, col, sfk)
    D = P.run_gpu(prob)
    P.check(prob, D, mode="exact")


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp8"])
@pytest.mark.parametrize("with_c", [False, True])
@pytest.mark.parametrize("kmul", [1, 4])
def test_block_scaled_pair_integers_bit_exact(kind, with_c, kmul):
    # 1000 x 2504: 40 tiles of 256 x 256 (CTA-pair instance), ragged in M and N; the
    # smallest legal K (NVFP4 256: one stage; MXFP8 512: four stages, one scale column)
    # and four times that
    K = (256 if kind == "nvfp4" else 512) * kmul
    prob = inputs.make_problem(kind, 1000, 2504, K, seed=15 + kmul, dist="int", with_c=with_c)
    P.check(prob, P.run_gpu(prob), mode="exact")


# ------------------------------------------------------------------ MXFP8

@pytest.mark.parametrize("with_c", [False, True])
@pytest.mark.parametrize("M", [128, 384])
def test_mxfp8_integers_bit_exact(with_c, M):
    # M = 384: CTA-pair instance (256-row tiles, the second one ragged), packed scales
    prob = inputs.make_problem("mxfp8", M, 256, 1024, seed=14, dist="int", with_c=with_c)
    P.check(prob, P.run_gpu(prob), mode="exact")


@pytest.mark.parametrize("M,N,K", [(300, 392, 1024), (128, 136, 512), (64, 2048, 4096), (2048, 4096, 2048)])
def test_mxfp8_random_tolerance(M, N, K):
    prob = inputs.make_problem("mxfp8", M, N, K, seed=M + N, dist="normal", with_c=True)
    P.check(prob, P.run_gpu(prob), mode="tol")


def test_mxfp8_8192_full_size_sampled_rows():
    # MXFP8 at the NVFP4 workload's size: CTA-pair instance, 32 x 32 tiles over 76 SM pairs
    prob = inputs.workload_problem("mxfp8_8192")
    D = P.run_gpu(prob)
    rows = P.sample_rows(prob["M"], 16, seed=4)
    P.check(prob, D, rows=rows, mode="tol")
    assert torch.isfinite(D.float()).all()


def test_nvfp4_8192_full_size_sampled_rows():
    prob = inputs.workload_problem("nvfp4_8192")
    D = P.run_gpu(prob)
    rows = P.sample_rows(prob["M"], 16, seed=3)
    P.check(prob, D, rows=rows, mode="tol")
    assert torch.isfinite(D.float()).all()


def test_mxfp8_128x16384_full_size_sampled_rows():
    prob = inputs.workload_problem("mxfp8_128x16384")
    D = P.run_gpu(prob)
    rows = P.sample_rows(prob["M"], 16, seed=4)
    P.check(prob, D, rows=rows, mode="tol")
    assert torch.isfinite(D.float()).all()


def test_fp16_pairs_partial_backward_raster_group():
    # 21 rows of 256 x 256 pair tiles run as raster groups of 16 and 5 m blocks; the
    # second (odd) group sweeps the columns backwards and is cut short
    M, N, K = 5376, 1024, 256
    sms = torch.cuda.get_device_properties(P.device()).multi_processor_count
    plan = P.dispatch_plan(M, N, K, 64, sms)
    assert plan[3] == 0 and plan[6] == 16, "not a CTA-pair launch with raster groups of 16"
    prob = inputs.make_problem("f16", M, N, K, seed=61, dist="int2", with_c=True)
    rows = [0, 255, 4095, 4096, 4100, 4351, 4352, 5000, 5375] + P.sample_rows(M, 16, seed=8)
    P.check(prob, P.run_gpu(prob, accum=0), rows=sorted(set(rows)), mode="exact")


# ------------------------------------------------------------------ split schedules
# Skinny shapes with long K, whose whole tiles would leave most of the device idle:
# the fp32 kinds give each tile to a cluster of up to 8 CTAs that split its k-blocks
# and add their fp32 partials through distributed shared memory.  Integer-valued
# inputs keep every fp32 partial sum exact, so the piecewise sum must match bit for
# bit.

@pytest.mark.parametrize("M,N,K,with_c", [(128, 2560, 16384, True), (500, 760, 16384, True),
                                          (64, 2056, 24576, False), (1, 4096, 16384, True)])
def test_split_fp16_integers_bit_exact(M, N, K, with_c):
    prob = inputs.make_problem("f16", M, N, K, seed=M + N + K, dist="int2", with_c=with_c)
    P.check(prob, P.run_gpu(prob, accum=0), rows=P.sample_rows(M, 24, seed=1), mode="exact")


# The reduction cuts each CTA's owned chunks into 1, 2 or 4 column parts, as the
# cluster size leaves room: clusters of 3 over 128 x 256 tiles (6 or 5 owned 32 x 64
# chunks: whole chunks per warp), and over 128 x 128 tiles clusters of 3 (3 or 2:
# halves), 4 (2: quarters) and 8 (1: quarters, half the warps idle).  The expected
# cluster sizes are the dispatch rules' on a 152-SM device.
@pytest.mark.parametrize("M,N,K,split", [(512, 2560, 8192, 3), (256, 2560, 16384, 3), (128, 4096, 4096, 4),
                                         (200, 1000, 32768, 8)])
def test_split_reduce_parts_fp16_integers_bit_exact(M, N, K, split):
    sms = torch.cuda.get_device_properties(P.device()).multi_processor_count
    plan = P.dispatch_plan(M, N, K, 64, sms)
    assert plan[4] > 1, "the shape no longer takes a cluster split"
    if sms == 152:
        assert plan[4] == split
    prob = inputs.make_problem("f16", M, N, K, seed=M + 7 * N + K, dist="int2", with_c=True)
    P.check(prob, P.run_gpu(prob, accum=0), rows=P.sample_rows(M, 32, seed=7), mode="exact")


# Stages of two 128-byte boxes of K: when K ends inside a stage, its second box lies
# partly (K = 8200: 8 of 64 elements) or wholly (K = 16448, 32840, 4160) past the end of
# K and is zero-filled; the split shares count whole stages.
@pytest.mark.parametrize("M,N,K", [(128, 2560, 16448), (200, 1000, 32840), (1024, 1024, 4160), (384, 520, 8200)])
def test_split_two_box_stages_ragged_k_bit_exact(M, N, K):
    sms = torch.cuda.get_device_properties(P.device()).multi_processor_count
    plan = P.dispatch_plan(M, N, K, 64, sms)
    assert plan[3] == 2 and plan[4] > 1, "not a split launch on 128 x 128 tiles"
    prob = inputs.make_problem("f16", M, N, K, seed=M + 3 * N + K, dist="int2", with_c=True)
    P.check(prob, P.run_gpu(prob, accum=0), rows=P.sample_rows(M, 24, seed=9), mode="exact")


def test_split_fp16_in_place():
    prob = inputs.make_problem("f16", 300, 520, 16384, seed=21, dist="int2", with_c=True)
    g = P.to_device(prob, P.device())
    D = g["C"].clone()
    tg.gemm_f16(g["A"], g["B"], D, D, tg.GEMM_ACC_F32)
    torch.cuda.synchronize()
    P.check(prob, D.cpu(), rows=P.sample_rows(300, 24, seed=6), mode="exact")


@pytest.mark.parametrize("M,N,K", [(1000, 1000, 16384), (129, 264, 65536)])
def test_split_fp16_random_tolerance(M, N, K):
    prob = inputs.make_problem("f16", M, N, K, seed=M + K, dist="normal0.1", with_c=True)
    P.check(prob, P.run_gpu(prob, accum=0), rows=P.sample_rows(M, 24, seed=2), mode="tol")


def test_split_repeatable_across_calls_and_streams():
    # a cluster adds its partials in rank order: the result depends on neither the call
    # nor the stream
    prob = inputs.make_problem("f16", 500, 760, 16384, seed=22, dist="normal0.1", with_c=True)
    first = P.run_gpu(prob, accum=0)
    s = torch.cuda.Stream()
    for stream in (None, s, None):
        again = P.run_gpu(prob, accum=0, stream=stream)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("M,N,K,with_c", [(128, 2048, 65536, True), (100, 3000, 65536, False)])
def test_split_nvfp4_integers_bit_exact(M, N, K, with_c):
    prob = inputs.make_problem("nvfp4", M, N, K, seed=M + N, dist="int", with_c=with_c)
    P.check(prob, P.run_gpu(prob), rows=P.sample_rows(M, 12, seed=3), mode="exact")


@pytest.mark.parametrize("M,N,K,with_c", [(100, 2048, 24576, True), (128, 1928, 24576, False)])
def test_split_mxfp8_integers_bit_exact(M, N, K, with_c):
    prob = inputs.make_problem("mxfp8", M, N, K, seed=M + N, dist="int", with_c=with_c)
    P.check(prob, P.run_gpu(prob), rows=P.sample_rows(M, 12, seed=4), mode="exact")


def test_split_mxfp8_random_tolerance():
    prob = inputs.make_problem("mxfp8", 128, 1024, 49152, seed=23, dist="normal", with_c=True)
    P.check(prob, P.run_gpu(prob), rows=P.sample_rows(128, 12, seed=5), mode="tol")


# ------------------------------------------------------------------ large extents
# One very long dimension at a time (the ABI takes each of M, N, K below 2^31; these
# stay within a few hundred MB of device memory).  Integer inputs keep every fp32
# partial sum exact, so sampled rows must match bit for bit.

def test_large_k_fp16_single_tile_split_over_a_cluster():
    # K = 2^20: one 128 x 128 tile whose 16384 k-blocks are split over a cluster of 8 CTAs
    prob = inputs.make_problem("f16", 128, 128, 1 << 20, seed=51, dist="int2", with_c=True)
    P.check(prob, P.run_gpu(prob, accum=0), rows=[0, 1, 63, 127], mode="exact")


def test_large_m_fp16_narrow_k():
    prob = inputs.make_problem("f16", 1 << 20, 16, 16, seed=52, dist="int2", with_c=True)
    D = P.run_gpu(prob, accum=0)
    P.check(prob, D, rows=P.sample_rows(1 << 20, 24, seed=5), mode="exact")


def test_large_n_fp16():
    prob = inputs.make_problem("f16", 128, 1 << 20, 32, seed=53, dist="int2", with_c=False)
    D = P.run_gpu(prob, accum=0)
    P.check(prob, D, rows=[0, 77, 127], mode="exact")


def test_large_k_nvfp4():
    prob = inputs.make_problem("nvfp4", 128, 256, 1 << 18, seed=54, dist="int", with_c=True)
    P.check(prob, P.run_gpu(prob), rows=[0, 31, 127], mode="exact")


# ------------------------------------------------------------------ argument errors on the GPU

def test_misaligned_output_is_rejected_not_faulted():
    dev = P.device()
    A = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    B = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    buf = torch.zeros(64 * 64 + 8, dtype=torch.float16, device=dev)
    D = buf[1:1 + 64 * 64].view(64, 64)
    with pytest.raises(tg.GemmError) as ei:
        tg.gemm_f16(A, B, None, D)
    assert ei.value.code == tg.GEMM_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert tg.gemm_last_device_error() == tg.GEMM_OK
