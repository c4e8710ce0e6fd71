"""gemm_f16_noalloc: the FP16 GEMM for callers that cannot allocate device memory.

Some callers may not allocate while they run: a plugin that may only use the
buffers its host application hands it, or a serving loop that reserved nearly
all of HBM in advance.  gemm_f16_noalloc never allocates: it runs skinny,
long-K problems on the stream-K schedule (every SM takes an equal share of the
k-blocks of the last tiles; the finishing unit adds the others' fp32 partials),
whose partials and flags live in a fixed block inside the loaded module.  These
tests call it through the C ABI:

  * on integer inputs, where every fp32 partial sum is exact, sampled rows must
    match the oracle bit for bit, on the stream-K shape (the host-side dispatch
    rule is checked to give that shape a split at the device's SM count) and on
    narrow K (16 and 32, one k-block: no split, no scratch);
  * on random inputs it must agree with gemm_f16 within the fp32-accumulation
    tolerance, on the stream-K shape and on a square whole-tile shape;

each twice in a row: the second call finds the first call's partials and flags
still in the shared block and must not be affected by them.

This file sorts last so that it also runs after every other GPU test; it needs
no state from them and passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import cute_layouts_mma_gb300 as tg
from cute_layouts_mma_gb300 import inputs

import _parity as P

pytestmark = pytest.mark.gpu


def _noalloc(g, D, stream):
    M, K = g["A"].shape
    N = g["B"].shape[0]
    C = g.get("C")
    return tg.lib().gemm_f16_noalloc(M, N, K, g["A"].data_ptr(), g["B"].data_ptr(),
                                     None if C is None else C.data_ptr(), D.data_ptr(),
                                     ctypes.c_void_p(stream.cuda_stream))


def _f16(g, D, stream):
    M, K = g["A"].shape
    N = g["B"].shape[0]
    C = g.get("C")
    return tg.lib().gemm_f16(M, N, K, g["A"].data_ptr(), g["B"].data_ptr(),
                             None if C is None else C.data_ptr(), D.data_ptr(), tg.GEMM_ACC_F32,
                             ctypes.c_void_p(stream.cuda_stream))


# 128 x 2560 x 16384 on the fixed-scratch call: the 128 x 256 tiles would split, so it
# takes the 128 x 128 single-CTA instance (20 tiles) with the stream-K schedule.
SPLIT_SHAPE = (128, 2560, 16384)


def test_noalloc_stream_k_integers_bit_exact_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = P.device()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    choice, split = P.dispatch_plan(*SPLIT_SHAPE, 64, sms)[:2]
    assert (choice, split) == (2, 1), "the shape no longer takes the stream-K schedule on this device"
    stream = torch.cuda.current_stream(dev)
    M, N, K = SPLIT_SHAPE
    for call, seed in enumerate((71, 72)):  # two calls in a row, different data
        prob = inputs.make_problem("f16", M, N, K, seed=seed, dist="int2", with_c=call == 0)
        g = P.to_device(prob, dev)
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert _noalloc(g, D, stream) == tg.GEMM_OK
        torch.cuda.synchronize(dev)
        assert tg.gemm_last_device_error() == tg.GEMM_OK
        P.check(prob, D.cpu(), rows=P.sample_rows(M, 24, seed=call), mode="exact")


@pytest.mark.parametrize("M,N,K", [(300, 264, 32), (128, 520, 16)])
def test_noalloc_narrow_k_integers_bit_exact(M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = P.device()
    stream = torch.cuda.current_stream(dev)
    for call in range(2):
        prob = inputs.make_problem("f16", M, N, K, seed=73 + call, dist="int2", with_c=True)
        g = P.to_device(prob, dev)
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert _noalloc(g, D, stream) == tg.GEMM_OK
        torch.cuda.synchronize(dev)
        assert tg.gemm_last_device_error() == tg.GEMM_OK
        P.check(prob, D.cpu(), mode="exact")


@pytest.mark.parametrize("M,N,K", [SPLIT_SHAPE, (1024, 1024, 1024)])
def test_noalloc_matches_gemm_f16_twice(M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = P.device()
    stream = torch.cuda.current_stream(dev)
    for call, seed in enumerate((41, 42)):  # two calls in a row, different data
        prob = inputs.make_problem("f16", M, N, K, seed=seed + M, dist="normal0.1", with_c=call == 0)
        g = P.to_device(prob, dev)
        D_ref = torch.empty(M, N, dtype=torch.float16, device=dev)
        D_new = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert _f16(g, D_ref, stream) == tg.GEMM_OK
        assert _noalloc(g, D_new, stream) == tg.GEMM_OK
        torch.cuda.synchronize(dev)
        assert tg.gemm_last_device_error() == tg.GEMM_OK
        ref = D_ref.cpu().double().numpy()
        new = D_new.cpu().double().numpy()
        assert not np.isnan(new).any(), f"call {call}: output not fully written"
        # the tolerance of the fp32-accumulation parity tests, plus one output ulp
        # for the two results' independent roundings (different split schedules)
        lim = P.tolerance_f32acc(prob) + 2 * P.half_ulp(ref, "f16")
        err = np.abs(new - ref)
        assert (err <= lim).all(), f"call {call}: max |diff| {err.max()} over tolerance"
