"""Layout-faithful emulations of one MMA.  TEST INFRASTRUCTURE ONLY.

They rebuild a product from operands placed where the pages say the hardware
expects them, so that the pages' placement rules can be checked against the
plain GEMM definition of the oracle.
"""
from __future__ import annotations

import numpy as np

from . import layouts as L


def sm80_m16n8k16_from_fragments(A: np.ndarray, B: np.ndarray, C: np.ndarray) -> np.ndarray:
    """D = A x B + C for one m16n8k16 TN MMA, via per-lane fragments.

    A is 16x16 (M,K), B is 8x16 (N,K), C is 16x8.  Operands are first scattered
    into 32 lanes x 8 (A) / 4 (B) slots by the (lane,value) -> (m,k) / (n,k)
    maps of "CuTe 中 A、B 如何加载到 MMA 寄存器" sections 2 and 5; each product term
    is then read back from the slot the inverse maps of the same sections
    name.  Any disagreement between forward and inverse maps, or a map that is
    not a bijection onto the tile, changes the result.
    """
    a_frag = np.full((32, 8), np.nan)
    b_frag = np.full((32, 4), np.nan)
    for t in range(32):
        for v in range(8):
            m, k = L.sm80_A_tv_to_mk(t, v)
            a_frag[t, v] = A[m, k]
        for v in range(4):
            n, k = L.sm80_B_tv_to_nk(t, v)
            b_frag[t, v] = B[n, k]
    D = np.array(C, dtype=np.float64, copy=True)
    for m in range(16):
        for n in range(8):
            acc = 0.0
            for k in range(16):
                ta, va = L.sm80_A_mk_to_tv(m, k)
                tb, vb = L.sm80_B_nk_to_tv(n, k)
                acc += a_frag[ta, va] * b_frag[tb, vb]
            D[m, n] += acc
    return D


def block_scaled_mma_via_tmem(a_val: np.ndarray, sfa_val: np.ndarray, b_val: np.ndarray,
                              sfb_val: np.ndarray, k_blk: int) -> np.ndarray:
    """One 128 x 128 x (4*k_blk) block-scaled MMA with its scales read from a TMEM model.

    a_val, b_val: decoded low-precision values, 128 x K each (rows m and n).
    sfa_val, sfb_val: decoded scales, 128 x 4.  The scales are first written to
    a 128-lane TMEM model through the base-tile packing and .warpx4 replication of
    "数据布局及其记号" (block-scaled section); row m of D is computed by lane
    partition p = m // 32, which reads SFA at (TLane m, TCol m//32, byte sfk)
    and SFB for column n at (TLane 32p + n%32, TCol n//32, byte sfk).
    """
    K = a_val.shape[1]
    assert K == 4 * k_blk
    tmem_a, tmem_b = {}, {}
    for r in range(128):
        for sfk in range(4):
            for loc in L.sf_tmem_locations(r, sfk):
                tmem_a[loc] = sfa_val[r, sfk]
                tmem_b[loc] = sfb_val[r, sfk]
    D = np.zeros((128, 128))
    for m in range(128):
        p = m // 32
        for n in range(128):
            acc = 0.0
            for k in range(K):
                sfk = k // k_blk
                sa = tmem_a[(m, m // 32, sfk)]
                sb = tmem_b[(32 * p + n % 32, n // 32, sfk)]
                acc += a_val[m, k] * sa * b_val[n, k] * sb
            D[m, n] = acc
    return D
