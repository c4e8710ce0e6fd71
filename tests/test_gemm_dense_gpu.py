"""GPU parity of the BF16 and unscaled FP8 TN GEMMs against the CPU oracle, through the C ABI."""
import pytest
import torch

import cute_layouts_mma_gb300 as tg
from cute_layouts_mma_gb300 import inputs

import _parity as P

pytestmark = pytest.mark.gpu

FP8 = ["fp8e4m3", "fp8e5m2"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tg.lib()


# ------------------------------------------------------------------ BF16

@pytest.mark.parametrize("M,N,K,with_c", [(384, 520, 512, True), (100, 264, 512, False), (256, 256, 256, True)])
def test_bf16_integers_bit_exact(M, N, K, with_c):
    prob = inputs.make_problem("bf16", M, N, K, seed=M + N + K, dist="int2", with_c=with_c)
    P.check(prob, P.run_gpu(prob), mode="exact")


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (130, 264, 72), (300, 520, 200), (257, 8, 1000),
                                   (64, 1000, 4096), (1000, 16, 520)])
def test_bf16_ragged_shapes_tolerance(M, N, K):
    prob = inputs.make_problem("bf16", M, N, K, seed=M + 2 * N + K, dist="normal0.1", with_c=True)
    P.check(prob, P.run_gpu(prob), mode="tol")


def test_bf16_in_place():
    prob = inputs.make_problem("bf16", 200, 264, 136, seed=31, dist="int2", with_c=True)
    g = P.to_device(prob, P.device())
    D = g["C"].clone()
    tg.gemm_bf16(g["A"], g["B"], D, D)
    torch.cuda.synchronize()
    P.check(prob, D.cpu(), mode="exact")


def test_bf16_split_integers_bit_exact():
    # a few tiles for a 152-SM device, 256 k-blocks: each tile split over a cluster of CTAs
    prob = inputs.make_problem("bf16", 128, 2560, 16384, seed=32, dist="int2", with_c=True)
    P.check(prob, P.run_gpu(prob), rows=P.sample_rows(128, 16, seed=1), mode="exact")


def test_bf16_4096_full_size_sampled_rows():
    prob = inputs.workload_problem("bf16_4096")
    D = P.run_gpu(prob)
    P.check(prob, D, rows=P.sample_rows(prob["M"], 16, seed=2), mode="tol")
    assert torch.isfinite(D.float()).all()


# ------------------------------------------------------------------ FP8 (no scales)

@pytest.mark.parametrize("kind", FP8)
@pytest.mark.parametrize("M,N,K,with_c", [(256, 264, 1024, True), (100, 512, 512, False), (512, 256, 2048, True)])
def test_fp8_integers_bit_exact(kind, M, N, K, with_c):
    prob = inputs.make_problem(kind, M, N, K, seed=M + N, dist="int", with_c=with_c)
    P.check(prob, P.run_gpu(prob), mode="exact")


@pytest.mark.parametrize("kind", FP8)
@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (130, 264, 96), (257, 8, 1008), (64, 1000, 4096), (300, 392, 1024)])
def test_fp8_ragged_shapes_tolerance(kind, M, N, K):
    prob = inputs.make_problem(kind, M, N, K, seed=M + 3 * N + K, dist="normal", with_c=True)
    P.check(prob, P.run_gpu(prob), mode="tol")


@pytest.mark.parametrize("kind", FP8)
def test_fp8_split_integers_bit_exact(kind):
    # a few tiles, 256 k-blocks of 128: each tile split over a cluster of CTAs
    prob = inputs.make_problem(kind, 128, 2048, 32768, seed=33, dist="int", with_c=True)
    P.check(prob, P.run_gpu(prob), rows=P.sample_rows(128, 12, seed=3), mode="exact")


def test_fp8e4m3_8192_full_size_sampled_rows():
    prob = inputs.workload_problem("fp8e4m3_8192")
    D = P.run_gpu(prob)
    P.check(prob, D, rows=P.sample_rows(prob["M"], 12, seed=4), mode="tol")
    assert torch.isfinite(D.float()).all()


# ------------------------------------------------------------------ in place, guard bands, concurrency

@pytest.mark.parametrize("kind,M,N,K", [("nvfp4", 300, 264, 1024), ("mxfp8", 200, 256, 1024), ("fp8e4m3", 300, 264, 1024),
                                        ("nvfp4", 1000, 2504, 512), ("mxfp8", 1000, 2504, 512)])
def test_in_place_d_is_c(kind, M, N, K):
    # 1000 x 2504: 40 tiles of 256 x 256, the block-scaled CTA-pair instance
    prob = inputs.make_problem(kind, M, N, K, seed=61, dist="int", with_c=True)
    g = P.to_device(prob, P.device())
    D = g["C"].clone()
    if kind == "fp8e4m3":
        tg.gemm_fp8(g["A"], g["B"], D, D, tg.GEMM_FP8_E4M3)
    else:
        fmt = tg.GEMM_FMT_NVFP4 if kind == "nvfp4" else tg.GEMM_FMT_MXFP8
        tg.gemm_block_scaled(g["A"], g["SFA"], g["B"], g["SFB"], D, D, fmt)
    torch.cuda.synchronize()
    P.check(prob, D.cpu(), mode="exact")


@pytest.mark.parametrize("kind,M,N,K", [("nvfp4", 130, 264, 512), ("fp8e5m2", 129, 136, 1008), ("bf16", 257, 8, 72),
                                        ("mxfp8", 1000, 2504, 512)])
def test_guard_bands_untouched(kind, M, N, K):
    # D sits between NaN guard bands; ragged M and N must not write outside it
    prob = inputs.make_problem(kind, M, N, K, seed=62, dist="int" if kind != "bf16" else "int2", with_c=True)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), float("nan"), dtype=torch.bfloat16, device=P.device())
    D = buf[pad:pad + M * N].view(M, N)
    P.run_gpu(prob, D=D)
    host = buf.cpu()
    assert torch.isnan(host[:pad].float()).all() and torch.isnan(host[pad + M * N:].float()).all()
    P.check(prob, D.cpu(), mode="exact")


def test_concurrent_split_calls_on_two_streams():
    # two split launches in flight at once on two streams: a split keeps its partials in
    # its own clusters' shared memory, so concurrent calls share nothing
    probs = [inputs.make_problem("f16", 128, 2560, 16384, seed=63 + i, dist="int2", with_c=True) for i in range(2)]
    dev = P.device()
    gs = [P.to_device(p, dev) for p in probs]
    Ds = [torch.empty(128, 2560, dtype=torch.float16, device=dev) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for rep in range(3):
        for g, D, s in zip(gs, Ds, streams):
            tg.gemm_f16(g["A"], g["B"], g["C"], D, tg.GEMM_ACC_F32, s)
    torch.cuda.synchronize()
    assert tg.gemm_last_device_error() == tg.GEMM_OK
    for p, D in zip(probs, Ds):
        P.check(p, D.cpu(), rows=P.sample_rows(128, 16, seed=8), mode="exact")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float8_e4m3fn, torch.float8_e5m2])
def test_gemm_dtype_dispatch(dtype):
    kind = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float8_e4m3fn: "fp8e4m3",
            torch.float8_e5m2: "fp8e5m2"}[dtype]
    prob = inputs.make_problem(kind, 200, 264, 256, seed=71, dist="int" if kind.startswith("fp8") else "int2",
                               with_c=True)
    g = P.to_device(prob, P.device())
    A, B = (g["A"].view(dtype), g["B"].view(dtype)) if kind.startswith("fp8") else (g["A"], g["B"])
    D = tg.gemm(A, B, g["C"])
    torch.cuda.synchronize()
    P.check(prob, D.cpu(), mode="exact")


# ------------------------------------------------------------------ instance choice by size

# Short-K problems whose 256-column tiles would keep fewer than half of the units busy take
# 128 x 64 tiles (most of the small shapes above); these sizes keep the 256-column tiles:
# 1000 x 2504 (40 CTA-pair tiles) and 120 x 19600 (77 single-CTA tiles), ragged edges.
@pytest.mark.parametrize("kind", ["f16", "bf16", "fp8e4m3"])
@pytest.mark.parametrize("M,N,K", [(1000, 2504, 512), (120, 19600, 256)])
def test_big_tile_sizes_bit_exact(kind, M, N, K):
    prob = inputs.make_problem(kind, M, N, K, seed=M + N + K, dist="int" if kind == "fp8e4m3" else "int2",
                               with_c=True)
    D = P.run_gpu(prob, accum=0) if kind == "f16" else P.run_gpu(prob)
    P.check(prob, D, mode="exact")
