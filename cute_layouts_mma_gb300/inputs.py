"""Seeded synthetic inputs for the TN GEMM workloads.

This module only draws random operands; it holds none of the GEMM's arithmetic.
It is the one piece shared by the CUDA path's tests/benchmark and the CPU
oracle's checks, so that both see the same bytes.  Everything is generated on
the CPU with torch.Generator(seed) and returned as CPU tensors.

Workloads (name -> recipe):
  fp16_int_256        M=N=K=256, A,B integers uniform in {-2..2} as half, C absent,
                      fp32 accumulation, fp16 D; every sum is exact.       seed 0
  fp16_4096           M=N=K=4096, A,B ~ N(0,1)*0.1 as half, C ~ N(0,1) half,
                      fp32 accumulation, fp16 D.                           seed 1
  fp16acc_8192x1024   M=N=8192, K=1024, A,B ~ U[-0.5,0.5] as half, C absent,
                      fp16 accumulation, fp16 D.                           seed 2
  nvfp4_8192          M=N=K=8192, E2M1 codes uniform over all 16, E4M3 scales
                      2^u with u uniform in {-3..3} (byte 0x38+8u), C absent,
                      fp32 accumulation, bf16 D.                           seed 3
  mxfp8_128x16384     M=128, N=16384, K=8192, E4M3 = RNE(clip(N(0,1), +-448)),
                      E8M0 exponents 127+U{-4..4}, C ~ N(0,1) bf16,
                      fp32 accumulation, bf16 D.                           seed 4
  bf16_4096           M=N=K=4096, A,B ~ N(0,1)*0.1 as bf16, C ~ N(0,1) bf16,
                      fp32 accumulation, bf16 D.                           seed 5
  fp8e4m3_8192        M=N=K=8192, A,B = E4M3 RNE(clip(N(0,1), +-448)), no
                      scales, C absent, fp32 accumulation, bf16 D.         seed 6
  mxfp8_8192          M=N=K=8192, as mxfp8_128x16384, C absent.            seed 7
  fp16_128x4096x4096  M=128, N=K=4096 (a skinny problem: each tile split over a
                      cluster), as fp16_4096 without C.                    seed 8
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

KIND_F16 = "f16"
KIND_NVFP4 = "nvfp4"
KIND_MXFP8 = "mxfp8"
KIND_BF16 = "bf16"
KIND_FP8_E4M3 = "fp8e4m3"
KIND_FP8_E5M2 = "fp8e5m2"
FP8_KINDS = (KIND_FP8_E4M3, KIND_FP8_E5M2)


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str          # "f16", "nvfp4", "mxfp8", "bf16", "fp8e4m3" or "fp8e5m2"
    M: int
    N: int
    K: int
    dist: str          # value recipe, see make_problem
    with_c: bool
    accum: int         # 0 = fp32, 1 = fp16 (FP16 kind only)
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    w.name: w for w in [
        Workload("fp16_int_256", KIND_F16, 256, 256, 256, "int2", False, 0, 0),
        Workload("fp16_4096", KIND_F16, 4096, 4096, 4096, "normal0.1", True, 0, 1),
        Workload("fp16acc_8192x1024", KIND_F16, 8192, 8192, 1024, "uniform0.5", False, 1, 2),
        Workload("nvfp4_8192", KIND_NVFP4, 8192, 8192, 8192, "codes", False, 0, 3),
        Workload("mxfp8_128x16384", KIND_MXFP8, 128, 16384, 8192, "normal", True, 0, 4),
        Workload("bf16_4096", KIND_BF16, 4096, 4096, 4096, "normal0.1", True, 0, 5),
        Workload("fp8e4m3_8192", KIND_FP8_E4M3, 8192, 8192, 8192, "normal", False, 0, 6),
        Workload("mxfp8_8192", KIND_MXFP8, 8192, 8192, 8192, "normal", False, 0, 7),
        Workload("fp16_128x4096x4096", KIND_F16, 128, 4096, 4096, "normal0.1", False, 0, 8),
    ]
}


def make_problem(kind: str, M: int, N: int, K: int, seed: int, dist: str = "default",
                 with_c: bool = True) -> dict:
    """Random operands for one GEMM, as CPU tensors.

    bf16:  as f16 with bfloat16 A, B, C ("int2" or "normal0.1").
    fp8e4m3 / fp8e5m2: A uint8[M,K], B uint8[N,K] FP8 codes (torch's RNE cast of
           clip(N(0,1)) to the format; "int": integers -4..4), C bf16 ~ N(0,1)
           ("int": integers -8..8) or None.
    f16:   A half[M,K], B half[N,K], C half[M,N] or None.  dist: "int2" (integers
           -2..2), "normal0.1" (N(0,1)*0.1), "uniform0.5" (U[-0.5,0.5]), "default"
           (= normal0.1).  C ~ N(0,1) when present ("int2": integers -50..50).
    nvfp4: A uint8[M,K/2] (random bytes: both nibbles uniform over the 16 E2M1
           codes), SFA uint8[M,K/16] = 0x38 + 8u, u ~ U{-3..3}; B, SFB likewise;
           "int" restricts codes to integer values and u to {0,1,2}.
           C bf16 ~ N(0,1) or None.
    mxfp8: A uint8[M,K] = E4M3 of clip(N(0,1), +-448) (torch's round-to-nearest-even
           cast), SFA uint8[M,K/32] = 127 + U{-4..4}; B, SFB likewise; "int"
           draws integer E4M3 values -4..4 and exponents 127 + U{0..2}.
           C bf16 ~ N(0,1) or None.
    """
    g = torch.Generator().manual_seed(seed)
    out: dict = {"kind": kind, "M": M, "N": N, "K": K}
    if kind == KIND_BF16:
        if dist == "int2":
            A = torch.randint(-2, 3, (M, K), generator=g).to(torch.bfloat16)
            B = torch.randint(-2, 3, (N, K), generator=g).to(torch.bfloat16)
            C = torch.randint(-50, 51, (M, N), generator=g).to(torch.bfloat16) if with_c else None
        else:
            A = (torch.randn(M, K, generator=g) * 0.1).to(torch.bfloat16)
            B = (torch.randn(N, K, generator=g) * 0.1).to(torch.bfloat16)
            C = torch.randn(M, N, generator=g).to(torch.bfloat16) if with_c else None
        out.update(A=A, B=B, C=C)
        return out
    if kind in FP8_KINDS:
        dt, lim = (torch.float8_e4m3fn, 448.0) if kind == KIND_FP8_E4M3 else (torch.float8_e5m2, 57344.0)
        if dist == "int":
            A = torch.randint(-4, 5, (M, K), generator=g).float().to(dt).view(torch.uint8)
            B = torch.randint(-4, 5, (N, K), generator=g).float().to(dt).view(torch.uint8)
            C = torch.randint(-8, 9, (M, N), generator=g).float().to(torch.bfloat16) if with_c else None
        else:
            A = torch.randn(M, K, generator=g).clamp(-lim, lim).to(dt).view(torch.uint8)
            B = torch.randn(N, K, generator=g).clamp(-lim, lim).to(dt).view(torch.uint8)
            C = torch.randn(M, N, generator=g).to(torch.bfloat16) if with_c else None
        out.update(A=A, B=B, C=C)
        return out
    if kind == KIND_F16:
        if dist == "int2":
            A = torch.randint(-2, 3, (M, K), generator=g).to(torch.float16)
            B = torch.randint(-2, 3, (N, K), generator=g).to(torch.float16)
            C = torch.randint(-50, 51, (M, N), generator=g).to(torch.float16) if with_c else None
        elif dist == "uniform0.5":
            A = (torch.rand(M, K, generator=g) - 0.5).to(torch.float16)
            B = (torch.rand(N, K, generator=g) - 0.5).to(torch.float16)
            C = torch.randn(M, N, generator=g).to(torch.float16) if with_c else None
        else:
            A = (torch.randn(M, K, generator=g) * 0.1).to(torch.float16)
            B = (torch.randn(N, K, generator=g) * 0.1).to(torch.float16)
            C = torch.randn(M, N, generator=g).to(torch.float16) if with_c else None
        out.update(A=A, B=B, C=C)
        return out
    if kind == KIND_NVFP4:
        if dist == "int":
            int_codes = torch.tensor([0, 2, 4, 5, 6, 7, 10, 12, 13, 14, 15], dtype=torch.uint8)
            ca = int_codes[torch.randint(0, len(int_codes), (M, K), generator=g)]
            cb = int_codes[torch.randint(0, len(int_codes), (N, K), generator=g)]
            A = (ca[:, 0::2] | (ca[:, 1::2] << 4)).contiguous()
            B = (cb[:, 0::2] | (cb[:, 1::2] << 4)).contiguous()
            u_lo, u_hi = 0, 2
        else:
            A = torch.randint(0, 256, (M, K // 2), generator=g, dtype=torch.uint8)
            B = torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.uint8)
            u_lo, u_hi = -3, 3
        SFA = (0x38 + 8 * torch.randint(u_lo, u_hi + 1, (M, K // 16), generator=g)).to(torch.uint8)
        SFB = (0x38 + 8 * torch.randint(u_lo, u_hi + 1, (N, K // 16), generator=g)).to(torch.uint8)
    elif kind == KIND_MXFP8:
        if dist == "int":
            A = torch.randint(-4, 5, (M, K), generator=g).float().to(torch.float8_e4m3fn).view(torch.uint8)
            B = torch.randint(-4, 5, (N, K), generator=g).float().to(torch.float8_e4m3fn).view(torch.uint8)
            e_lo, e_hi = 0, 2
        else:
            A = torch.randn(M, K, generator=g).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            B = torch.randn(N, K, generator=g).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            e_lo, e_hi = -4, 4
        SFA = (127 + torch.randint(e_lo, e_hi + 1, (M, K // 32), generator=g)).to(torch.uint8)
        SFB = (127 + torch.randint(e_lo, e_hi + 1, (N, K // 32), generator=g)).to(torch.uint8)
    else:
        raise ValueError(kind)
    if with_c:
        C = (torch.randint(-8, 9, (M, N), generator=g).float() if dist == "int"
             else torch.randn(M, N, generator=g)).to(torch.bfloat16)
    else:
        C = None
    out.update(A=A, SFA=SFA, B=B, SFB=SFB, C=C)
    return out


def workload_problem(name: str) -> dict:
    w = WORKLOADS[name]
    p = make_problem(w.kind, w.M, w.N, w.K, w.seed, w.dist, w.with_c)
    p["accum"] = w.accum
    return p
