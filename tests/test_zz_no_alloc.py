"""gemm_f16_noalloc: the FP16 GEMM for callers that cannot allocate device memory.

Some callers may not allocate while they run: a plugin that may only use the
buffers its host application hands it, or a serving loop that reserved nearly
all of HBM in advance.  For them the library offers gemm_f16_noalloc, which
keeps its stream-K scratch in a fixed block inside the loaded module instead of
taking it from a memory pool.  These tests call it through the C ABI and compare
it with gemm_f16 on a skinny, long-K shape (where the stream-K schedule and so
the scratch are used) and on a square shape (whole tiles, no scratch), twice in
a row each: the second call finds the first call's partials and flags still in
the shared block and must not be affected by them.

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


def _pooled(g, D, stream):
    M, K = g["A"].shape
    N = g["B"].shape[0]
    C = g.get("C")
    return tg.lib().gemm_f16(M, N, K, g["A"].data_ptr(), g["B"].data_ptr(),
                             None if C is None else C.data_ptr(), D.data_ptr(), tg.GEMM_ACC_F32,
                             ctypes.c_void_p(stream.cuda_stream))


# (M, N, K): 128 x 2560 x 16384 takes the stream-K schedule (10 tiles on a
# 152-SM device, each split between about 15 units); 1024^3 takes whole tiles.
@pytest.mark.parametrize("M,N,K", [(128, 2560, 16384), (1024, 1024, 1024)])
def test_noalloc_matches_pooled_entry_point_twice(M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = P.device()
    stream = torch.cuda.current_stream(dev)
    for call, seed in enumerate((41, 42)):  # two calls in a row, different data
        prob = inputs.make_problem("f16", M, N, K, seed=seed + M, dist="normal0.1", with_c=call == 0)
        g = P.to_device(prob, dev)
        D_ref = torch.empty(M, N, dtype=torch.float16, device=dev)
        D_new = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert _pooled(g, D_ref, stream) == tg.GEMM_OK
        assert _noalloc(g, D_new, stream) == tg.GEMM_OK
        torch.cuda.synchronize(dev)
        assert tg.gemm_last_device_error() == tg.GEMM_OK
        ref = D_ref.cpu().double().numpy()
        new = D_new.cpu().double().numpy()
        assert not np.isnan(new).any(), f"call {call}: output not fully written"
        # the tolerance of the fp32-accumulation parity tests, plus one output ulp
        # for the two results' independent roundings
        lim = P.tolerance_f32acc(prob) + 2 * P.half_ulp(ref, "f16")
        err = np.abs(new - ref)
        assert (err <= lim).all(), f"call {call}: max |diff| {err.max()} over tolerance"
