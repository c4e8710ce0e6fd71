"""Pins of the oracle GEMMs (CPU only): brute force in exact rationals, identity and
permutation operands, integer cases against numpy's matmul, and one-hot scale
probes that localise the block-scale indexing."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _f16(t):
    return t.to(torch.float16)


def _exact_f16_gemm(A, B, C):
    M, K = A.shape
    N = B.shape[0]
    a = [[Fraction(float(x)) for x in row] for row in A.double().tolist()]
    b = [[Fraction(float(x)) for x in row] for row in B.double().tolist()]
    c = [[Fraction(float(x)) for x in row] for row in C.double().tolist()] if C is not None else None
    out = [[(c[m][n] if c else 0) + sum(a[m][k] * b[n][k] for k in range(K)) for n in range(N)]
           for m in range(M)]
    return out


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (8, 2, 5), (4, 8, 8), (7, 7, 3)])
def test_f16_brute_force_exact_rationals(M, N, K):
    g = torch.Generator().manual_seed(M * 100 + N * 10 + K)
    A = _f16(torch.randn(M, K, generator=g))
    B = _f16(torch.randn(N, K, generator=g))
    C = _f16(torch.randn(M, N, generator=g))
    d16, d64 = oracle.gemm_f16(A, B, C, exact=True)
    ex = _exact_f16_gemm(A, B, C)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(d64[m, n]) - ex[m][n]) <= abs(ex[m][n]) * Fraction(1, 2 ** 50)
            want = np.array([float(ex[m][n])]).astype(np.float16).view(np.uint16)[0]
            assert d16[m, n] == want


def test_f16_identity_and_permutation():
    g = torch.Generator().manual_seed(3)
    n = 24
    B = _f16(torch.randn(n, n, generator=g))
    C = _f16(torch.randn(n, n, generator=g))
    I = torch.eye(n).half()
    # A = I: D[m][n] = sum_k I[m][k] B[n][k] = B[n][m]
    d = oracle.gemm_f16(I, B, None)
    assert np.array_equal(d, B.T.contiguous().view(torch.int16).numpy().view(np.uint16))
    # B = I: D = A + C  (one rounding of an exact sum)
    d = oracle.gemm_f16(B, I, C)
    want = (B.double() + C.double()).numpy().astype(np.float16).view(np.uint16)
    assert np.array_equal(d, want)
    # A = permutation P: D = rows of B^T permuted
    perm = torch.randperm(n, generator=g)
    P = torch.zeros(n, n).index_put_((torch.arange(n), perm), torch.ones(n)).half()
    d = oracle.gemm_f16(P, B, None)
    assert np.array_equal(d, B.T.contiguous()[perm].view(torch.int16).numpy().view(np.uint16))


def test_f16_small_integers_exact_vs_numpy():
    g = torch.Generator().manual_seed(0)
    M = N = K = 96
    A = torch.randint(-2, 3, (M, K), generator=g).half()
    B = torch.randint(-2, 3, (N, K), generator=g).half()
    C = torch.randint(-50, 51, (M, N), generator=g).half()
    want = (np.matmul(A.double().numpy(), B.double().numpy().T) + C.double().numpy())
    d = oracle.gemm_f16(A, B, C)
    assert np.array_equal(d, want.astype(np.float16).view(np.uint16))


def test_f16_row_subset_matches_full():
    g = torch.Generator().manual_seed(4)
    A = _f16(torch.randn(40, 33, generator=g))
    B = _f16(torch.randn(17, 33, generator=g))
    full = oracle.gemm_f16(A, B)
    rows = [39, 0, 7, 7, 21]
    assert np.array_equal(oracle.gemm_f16(A, B, rows=rows), full[rows])


# ---- block-scaled ---------------------------------------------------------------

def _e2m1_via_torch(codes: torch.Tensor) -> torch.Tensor:
    """Decode E2M1 codes by re-encoding them as E4M3 bytes and letting torch decode:
    exponent field e>0 -> e+6 with the mantissa bit moved to the top of 3; e=0
    (value m*0.5) -> 0 or the E4M3 code of 0.5."""
    c = codes.to(torch.int32)
    s, e, m = c >> 3, (c >> 1) & 3, c & 1
    mag = torch.where(e > 0, ((e + 6) << 3) | (m << 2), torch.where(m > 0, 6 << 3, 0))
    return ((s << 7) | mag).to(torch.uint8).view(torch.float8_e4m3fn).double()


def _pack_fp4(codes: torch.Tensor) -> torch.Tensor:
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()


def test_nvfp4_integer_case_vs_numpy():
    g = torch.Generator().manual_seed(21)
    M, N, K = 48, 40, 128
    # integer E2M1 magnitudes (0,1,2,3,4,6 and signs) with scales 2^u, u >= 0
    int_codes = torch.tensor([0, 2, 4, 5, 6, 7, 8 | 2, 8 | 4, 8 | 5, 8 | 6, 8 | 7], dtype=torch.uint8)
    a = int_codes[torch.randint(0, len(int_codes), (M, K), generator=g)]
    b = int_codes[torch.randint(0, len(int_codes), (N, K), generator=g)]
    sfa = (0x38 + 8 * torch.randint(0, 3, (M, K // 16), generator=g)).to(torch.uint8)
    sfb = (0x38 + 8 * torch.randint(0, 3, (N, K // 16), generator=g)).to(torch.uint8)
    C = torch.randint(-8, 9, (M, N), generator=g).to(torch.bfloat16)
    ar = _e2m1_via_torch(a) * sfa.view(torch.float8_e4m3fn).double().repeat_interleave(16, dim=1)
    br = _e2m1_via_torch(b) * sfb.view(torch.float8_e4m3fn).double().repeat_interleave(16, dim=1)
    want = np.matmul(ar.numpy(), br.numpy().T) + C.double().numpy()
    d16, d64 = oracle.gemm_block_scaled(oracle.NVFP4, _pack_fp4(a), sfa, _pack_fp4(b), sfb, C,
                                        exact=True)
    assert np.array_equal(d64, want)
    want16 = torch.from_numpy(want).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(d16, want16)  # |D| small integers: fp32 intermediate is exact


def test_mxfp8_case_vs_numpy():
    g = torch.Generator().manual_seed(22)
    M, N, K = 33, 29, 256
    a = torch.randn(M, K, generator=g).clamp(-448, 448).to(torch.float8_e4m3fn)
    b = torch.randn(N, K, generator=g).clamp(-448, 448).to(torch.float8_e4m3fn)
    sfa = (127 + torch.randint(-4, 5, (M, K // 32), generator=g)).to(torch.uint8)
    sfb = (127 + torch.randint(-4, 5, (N, K // 32), generator=g)).to(torch.uint8)
    C = torch.randn(M, N, generator=g).to(torch.bfloat16)
    ar = a.double() * sfa.view(torch.float8_e8m0fnu).double().repeat_interleave(32, dim=1)
    br = b.double() * sfb.view(torch.float8_e8m0fnu).double().repeat_interleave(32, dim=1)
    want = np.matmul(ar.numpy(), br.numpy().T) + C.double().numpy()
    d16, d64 = oracle.gemm_block_scaled(oracle.MXFP8, a.view(torch.uint8), sfa, b.view(torch.uint8),
                                        sfb, C, exact=True)
    assert np.allclose(d64, want, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP8])
def test_one_hot_scale_probe(fmt):
    """All data 1.0 and all scales 1 except SFA[row, sfk] = 2 (and, separately,
    SFB[col, sfk] = 2): only that row (column) of D changes, by exactly K_blk."""
    M, N, K = 64, 48, 256
    kblk = oracle.K_BLK[fmt]
    if fmt == oracle.NVFP4:
        one, s1, s2 = 0x2, 0x38, 0x40  # E2M1 1.0; E4M3 1.0 and 2.0
        A = torch.full((M, K // 2), one | (one << 4), dtype=torch.uint8)
        B = torch.full((N, K // 2), one | (one << 4), dtype=torch.uint8)
    else:
        one, s1, s2 = 0x38, 127, 128  # E4M3 1.0; E8M0 1.0 and 2.0
        A = torch.full((M, K), one, dtype=torch.uint8)
        B = torch.full((N, K), one, dtype=torch.uint8)
    SFA = torch.full((M, K // kblk), s1, dtype=torch.uint8)
    SFB = torch.full((N, K // kblk), s1, dtype=torch.uint8)
    row, col, sfk = 37, 11, 3
    SFA[row, sfk] = s2
    _, d = oracle.gemm_block_scaled(fmt, A, SFA, B, SFB, exact=True)
    want = np.full((M, N), float(K))
    want[row, :] += kblk
    assert np.array_equal(d, want)
    SFA[row, sfk] = s1
    SFB[col, sfk] = s2
    _, d = oracle.gemm_block_scaled(fmt, A, SFA, B, SFB, exact=True)
    want = np.full((M, N), float(K))
    want[:, col] += kblk
    assert np.array_equal(d, want)


def test_nvfp4_nibble_order_reading():
    """Element 2j is the low nibble of byte j (the stated packing reading)."""
    A = torch.tensor([[0x21] + [0] * 7], dtype=torch.uint8)   # elements: 0.5 (code 1), 1.0 (code 2)
    Bk0 = torch.tensor([[0x02] + [0] * 7], dtype=torch.uint8)  # B = one-hot 1.0 at k = 0
    Bk1 = torch.tensor([[0x20] + [0] * 7], dtype=torch.uint8)  # one-hot 1.0 at k = 1
    SF = torch.full((1, 1), 0x38, dtype=torch.uint8)
    _, d0 = oracle.gemm_block_scaled(oracle.NVFP4, A, SF, Bk0, SF, exact=True)
    _, d1 = oracle.gemm_block_scaled(oracle.NVFP4, A, SF, Bk1, SF, exact=True)
    assert d0[0, 0] == 0.5 and d1[0, 0] == 1.0


def test_block_scaled_rejects_ragged_k():
    A = np.zeros((2, 24), np.uint8)
    SF = np.zeros((2, 1), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_block_scaled(oracle.MXFP8, A, SF, A, SF)


# ---- dense GEMM over BF16 / FP8 operands ------------------------------------------

_TORCH = {oracle.FP16: torch.float16, oracle.BF16: torch.bfloat16,
          oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def _cast(x, fmt):
    return x.to(_TORCH[fmt])


def _exact_dense(A, B, C):
    """Exact rational sums of the decoded (torch) operand values."""
    a = [[Fraction(float(x)) for x in row] for row in A.double().tolist()]
    b = [[Fraction(float(x)) for x in row] for row in B.double().tolist()]
    c = [[Fraction(float(x)) for x in row] for row in C.double().tolist()] if C is not None else None
    return [[(c[m][n] if c else 0) + sum(a[m][k] * b[n][k] for k in range(len(a[0])))
             for n in range(len(b))] for m in range(len(a))]


@pytest.mark.parametrize("a_fmt,b_fmt,out_fmt", [(oracle.BF16, oracle.BF16, oracle.BF16),
                                                 (oracle.E4M3, oracle.E4M3, oracle.BF16),
                                                 (oracle.E5M2, oracle.E5M2, oracle.BF16),
                                                 (oracle.E4M3, oracle.E5M2, oracle.FP16)])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (6, 4, 16)])
def test_dense_brute_force_exact_rationals(a_fmt, b_fmt, out_fmt, M, N, K):
    g = torch.Generator().manual_seed(M * 100 + N * 10 + K + 7 * a_fmt + b_fmt)
    A = _cast(torch.randn(M, K, generator=g) * 2, a_fmt)
    B = _cast(torch.randn(N, K, generator=g) * 2, b_fmt)
    C = _cast(torch.randn(M, N, generator=g), out_fmt)
    d16, d64 = oracle.gemm_dense(A, B, C, a_fmt, b_fmt, out_fmt, exact=True)
    ex = _exact_dense(A, B, C)
    out_t = _TORCH[out_fmt]
    for m in range(M):
        for n in range(N):
            assert Fraction(d64[m, n]) == ex[m][n]  # products of <= 8-bit mantissas sum exactly here
            want = torch.tensor([float(ex[m][n])], dtype=torch.float64).to(out_t).view(torch.int16).item() & 0xFFFF
            assert d16[m, n] == want


@pytest.mark.parametrize("fmt,lo,hi", [(oracle.BF16, -8, 9), (oracle.E4M3, -8, 9), (oracle.E5M2, -4, 5)])
def test_dense_small_integers_exact_vs_numpy(fmt, lo, hi):
    g = torch.Generator().manual_seed(20 + fmt)
    M, N, K = 48, 40, 136
    A = torch.randint(lo, hi, (M, K), generator=g).float()
    B = torch.randint(lo, hi, (N, K), generator=g).float()
    C = torch.randint(-50, 51, (M, N), generator=g).float()
    want = np.matmul(A.double().numpy(), B.double().numpy().T) + C.double().numpy()
    d = oracle.gemm_dense(_cast(A, fmt), _cast(B, fmt), C.bfloat16(), fmt, fmt, oracle.BF16)
    assert np.array_equal(d, torch.from_numpy(want).bfloat16().view(torch.int16).numpy().view(np.uint16))


def test_dense_identity_permutation_and_fp16_agreement():
    g = torch.Generator().manual_seed(5)
    n = 32
    B = torch.randn(n, n, generator=g).to(torch.float8_e4m3fn)
    I = torch.eye(n).to(torch.float8_e4m3fn)
    val = lambda bits: oracle.bf16_bits_to_f64_array(bits)  # compares -0 equal to +0
    # A = I: D[m][n] = B[n][m], exact in bf16 (every E4M3 value is a bf16 value)
    d = oracle.gemm_dense(I, B, None, oracle.E4M3, oracle.E4M3, oracle.BF16)
    assert np.array_equal(val(d), B.T.double().numpy())
    perm = torch.randperm(n, generator=g)
    P = torch.zeros(n, n).index_put_((torch.arange(n), perm), torch.ones(n)).to(torch.float8_e4m3fn)
    d = oracle.gemm_dense(P, B, None, oracle.E4M3, oracle.E4M3, oracle.BF16)
    assert np.array_equal(val(d), B.T.contiguous()[perm].double().numpy())
    # fp16 operands and fp16 output: the same numbers as the FP16 oracle
    A16 = torch.randn(9, 20, generator=g).half()
    B16 = torch.randn(11, 20, generator=g).half()
    C16 = torch.randn(9, 11, generator=g).half()
    assert np.array_equal(oracle.gemm_dense(A16, B16, C16, oracle.FP16, oracle.FP16, oracle.FP16),
                          oracle.gemm_f16(A16, B16, C16))


def test_dense_rejects_unknown_format():
    A = np.zeros((2, 4), dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_dense(A, A, None, 7, oracle.E4M3, oracle.BF16)
    with pytest.raises(ValueError):
        oracle.gemm_dense(A, A, None, oracle.E4M3, oracle.E4M3, oracle.E4M3)
