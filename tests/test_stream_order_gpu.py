"""Back-to-back calls on one stream with no host synchronisation between them.

Every launch uses programmatic dependent launch: a kernel lets the next one on the
stream start its set-up early, and each thread of the next kernel waits for the
previous grid only right before its first global-memory access (the TMA issuers
before their first operand or scale load, the epilogue before its first C load or D
store).  These tests make the second call depend on the first through memory, while
the first is still long enough to be running when the second starts:

  * read after write: the second call reads the first call's D as its A operand, or,
    for NVFP4, as its SFA scale bytes;
  * write after read: the second call writes its D over the first call's A.

Integer-valued inputs keep every sum exact, so results are compared bit for bit
(the first call against the oracle, the second against the first call's output).
"""
import numpy as np
import pytest
import torch

import cute_layouts_mma_gb300 as tg
from cute_layouts_mma_gb300 import inputs

import _parity as P

pytestmark = pytest.mark.gpu


def _perm_matrix(n: int, seed: int, dev):
    """P [n][n] half with P[j, perm[j]] = 1: (X P^T)[:, j] = X[:, perm[j]]."""
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(seed))
    Pm = torch.zeros(n, n, dtype=torch.float16)
    Pm[torch.arange(n), perm] = 1.0
    return Pm.to(dev), perm


@pytest.mark.parametrize("M,N,K", [(512, 512, 256), (128, 4096, 4096), (2048, 2048, 4096)])
def test_read_after_write_fp16(M, N, K):
    # 128 x 64 tiles, a cluster split and CTA pairs for the first call
    dev = P.device()
    prob = inputs.make_problem("f16", M, N, K, seed=M + N + K, dist="int2", with_c=True)
    g = P.to_device(prob, dev)
    Pm, perm = _perm_matrix(N, seed=K, dev=dev)
    D1 = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    D2 = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    tg.gemm_f16(g["A"], g["B"], g["C"], D1, tg.GEMM_ACC_F32)
    tg.gemm_f16(D1, Pm, None, D2, tg.GEMM_ACC_F32)  # reads D1 as its A
    torch.cuda.synchronize(dev)
    assert tg.gemm_last_device_error() == tg.GEMM_OK
    d1 = D1.cpu()
    P.check(prob, d1, rows=P.sample_rows(M, 24, seed=11), mode="exact")
    assert torch.equal(D2.cpu().view(torch.int16), d1[:, perm].view(torch.int16))


def test_write_after_read_fp16():
    # the first call (CTA pairs, ~25 us) reads A; the second overwrites A at once
    dev = P.device()
    M, N, K = 2048, 2048, 4096
    prob = inputs.make_problem("f16", M, N, K, seed=31, dist="int2", with_c=False)
    g = P.to_device(prob, dev)
    over = inputs.make_problem("f16", M, K, 64, seed=32, dist="int2", with_c=False)
    go = P.to_device(over, dev)
    D1 = torch.empty(M, N, dtype=torch.float16, device=dev)
    tg.gemm_f16(g["A"], g["B"], None, D1, tg.GEMM_ACC_F32)
    tg.gemm_f16(go["A"], go["B"], None, g["A"], tg.GEMM_ACC_F32)  # D of the second call = A of the first
    torch.cuda.synchronize(dev)
    assert tg.gemm_last_device_error() == tg.GEMM_OK
    P.check(prob, D1.cpu(), rows=P.sample_rows(M, 24, seed=12), mode="exact")
    P.check(over, g["A"].cpu(), rows=P.sample_rows(M, 24, seed=13), mode="exact")


def test_read_after_write_nvfp4_scales():
    # The first call writes C unchanged (A = 0) into a buffer whose bytes the second call
    # (NVFP4, CTA pairs with the SFB multicast) reads as SFA; the bytes are valid scales
    # 1, 2 or 4, the buffer starts out holding scales of 1 everywhere.
    dev = P.device()
    M2, N2, K2 = 2048, 2048, 8192
    prob = inputs.make_problem("nvfp4", M2, N2, K2, seed=41, dist="int", with_c=False)
    sf_cols = K2 // 16
    gen = torch.Generator().manual_seed(42)
    sfa = (0x38 + 8 * torch.randint(0, 3, (M2, sf_cols), generator=gen)).to(torch.uint8)
    prob["SFA"] = sfa
    c1 = sfa.view(torch.float16)  # [M2][sf_cols / 2] half values with those bytes
    assert torch.isfinite(c1.float()).all()
    n1, k1 = sf_cols // 2, 8192
    A1 = torch.zeros(M2, k1, dtype=torch.float16, device=dev)
    B1 = torch.ones(n1, k1, dtype=torch.float16, device=dev)
    D1 = torch.full((M2, n1), 1.0, dtype=torch.float16, device=dev)
    D1.view(torch.uint8).fill_(0x38)
    g = P.to_device(prob, dev)
    D2 = torch.empty(M2, N2, dtype=torch.bfloat16, device=dev)
    tg.gemm_f16(A1, B1, c1.to(dev), D1, tg.GEMM_ACC_F32)
    tg.gemm_block_scaled(g["A"], D1.view(torch.uint8), g["B"], g["SFB"], None, D2, tg.GEMM_FMT_NVFP4)
    torch.cuda.synchronize(dev)
    assert tg.gemm_last_device_error() == tg.GEMM_OK
    assert torch.equal(D1.cpu().view(torch.uint8), sfa)
    P.check(prob, D2.cpu(), rows=P.sample_rows(M2, 12, seed=14), mode="exact")
