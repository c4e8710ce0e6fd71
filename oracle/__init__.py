"""CPU oracle for the TN GEMM D = A x B + C (FP16, BF16, FP8 and block-scaled NVFP4 / MXFP8).

TEST INFRASTRUCTURE ONLY.  This package is the independent checker of the CUDA
library: only the tests, the package smoke check and the benchmark's CPU-baseline
leg may import it.  The product path never imports, links or calls it, and it
shares no code with the CUDA sources.

Contents
  oracle.c   -- plain fp64 GEMM loops and the element decoders / output rounding
                ("CuTe 中 A、B 如何加载到 MMA 寄存器" section 1 for D = A x B + C in
                TN form; "数据布局及其记号", block-scaled MMA section, for the
                scaled operands).  Built with gcc into _build/liboracle.so.
  layouts.py -- the pages' layout functions (Shape:Stride, named axes, TV
                layouts, make_fragment_like, retile, swizzle, scale-factor TMEM
                placement) used to pin the oracle against the pages' worked
                examples.

Parity status: every function here is pinned by tests under tests/ marked
"not gpu" (page values, closed forms, torch/numpy decoders, brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")

NVFP4 = 0
MXFP8 = 1
K_BLK = {NVFP4: 16, MXFP8: 32}


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP over output rows, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        i64p = ctypes.POINTER(ctypes.c_int64)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        l.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        l.oracle_f16_to_f64.restype = ctypes.c_double
        l.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        l.oracle_bf16_to_f64.restype = ctypes.c_double
        for name in ("oracle_e2m1_to_f64", "oracle_e4m3_to_f64", "oracle_e5m2_to_f64", "oracle_e8m0_to_f64"):
            getattr(l, name).argtypes = [ctypes.c_uint8]
            getattr(l, name).restype = ctypes.c_double
        l.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        l.oracle_f64_to_f16.restype = ctypes.c_uint16
        l.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        l.oracle_f64_to_bf16.restype = ctypes.c_uint16
        l.oracle_gemm_f16.argtypes = [i64, i64, i64, u16p, u16p, u16p, i64p, i64, u16p, f64p]
        l.oracle_gemm_f16.restype = None
        l.oracle_gemm_block_scaled.argtypes = [ctypes.c_int, i64, i64, i64, u8p, u8p, u8p, u8p,
                                               u16p, i64p, i64, u16p, f64p]
        l.oracle_gemm_block_scaled.restype = ctypes.c_int
        vp = ctypes.c_void_p
        l.oracle_gemm_dense.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, i64, i64, vp, vp,
                                        u16p, i64p, i64, u16p, f64p]
        l.oracle_gemm_dense.restype = ctypes.c_int
        l.oracle_num_threads.argtypes = []
        l.oracle_num_threads.restype = ctypes.c_int
        _lib = l
    return _lib


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _bits16(x) -> np.ndarray:
    """Accept numpy uint16/float16 arrays or torch fp16/bf16 tensors; return uint16 bits."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    x = np.ascontiguousarray(x)
    return x.view(np.uint16)


def _bytes(x) -> np.ndarray:
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().contiguous().view(torch.uint8).numpy()
    return np.ascontiguousarray(x).view(np.uint8)


def num_threads() -> int:
    return lib().oracle_num_threads()


def gemm_f16(A, B, C=None, rows=None, exact: bool = False):
    """D = round_fp16(C + A @ B^T) for A fp16[M][K], B fp16[N][K] (TN), fp64 sums.

    rows: optional list of m indices; the result then has len(rows) rows.
    Returns uint16 fp16 bits [rows, N], plus the unrounded fp64 sums if exact.
    """
    A, B = _bits16(A), _bits16(B)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    Cb = None if C is None else _bits16(C)
    if Cb is not None:
        assert Cb.shape == (M, N)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nr = M if r is None else len(r)
    D16 = np.zeros((nr, N), dtype=np.uint16)
    D64 = np.zeros((nr, N), dtype=np.float64) if exact else None
    lib().oracle_gemm_f16(M, N, K, _ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16),
                          _ptr(Cb, ctypes.c_uint16), _ptr(r, ctypes.c_int64), nr,
                          _ptr(D16, ctypes.c_uint16), _ptr(D64, ctypes.c_double))
    return (D16, D64) if exact else D16


def gemm_block_scaled(fmt: int, A, SFA, B, SFB, C=None, rows=None, exact: bool = False):
    """D = round_bf16(C + A_real @ B_real^T), A_real = decode(A)*decode(SFA[m, k//K_blk]).

    fmt: NVFP4 (A u8[M][K/2], two E2M1 per byte, low nibble first; SFA E4M3
    u8[M][K/16]) or MXFP8 (A u8[M][K] E4M3; SFA E8M0 u8[M][K/32]).  B, SFB
    likewise with N rows.  C: bf16[M][N] bits or None.
    """
    A, SFA, B, SFB = _bytes(A), _bytes(SFA), _bytes(B), _bytes(SFB)
    M = A.shape[0]
    N = B.shape[0]
    K = A.shape[1] * (2 if fmt == NVFP4 else 1)
    Cb = None if C is None else _bits16(C)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nr = M if r is None else len(r)
    D16 = np.zeros((nr, N), dtype=np.uint16)
    D64 = np.zeros((nr, N), dtype=np.float64) if exact else None
    rc = lib().oracle_gemm_block_scaled(fmt, M, N, K, _ptr(A, ctypes.c_uint8),
                                        _ptr(SFA, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                                        _ptr(SFB, ctypes.c_uint8), _ptr(Cb, ctypes.c_uint16),
                                        _ptr(r, ctypes.c_int64), nr, _ptr(D16, ctypes.c_uint16),
                                        _ptr(D64, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle: K must be a multiple of the scale block and fmt 0 or 1")
    return (D16, D64) if exact else D16


# element formats of gemm_dense
FP16, BF16, E4M3, E5M2 = 0, 1, 2, 3


def _dense_operand(x, fmt: int) -> np.ndarray:
    return _bits16(x) if fmt in (FP16, BF16) else _bytes(x)


def gemm_dense(A, B, C=None, a_fmt: int = BF16, b_fmt: int = BF16, out_fmt: int = BF16, rows=None,
               exact: bool = False):
    """D = round_out(C + A @ B^T) for A a_fmt[M][K], B b_fmt[N][K] (TN), fp64 sums.

    Formats: FP16 / BF16 (torch half / bfloat16 tensors or uint16 bit arrays),
    E4M3 / E5M2 (torch float8 tensors or uint8 code arrays).  C and D are out_fmt
    (FP16 or BF16) bits.  Returns uint16 bits [rows, N] (plus the fp64 sums if exact).
    """
    Ab, Bb = _dense_operand(A, a_fmt), _dense_operand(B, b_fmt)
    M, K = Ab.shape
    N, K2 = Bb.shape
    assert K == K2
    Cb = None if C is None else _bits16(C)
    if Cb is not None:
        assert Cb.shape == (M, N)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nr = M if r is None else len(r)
    D16 = np.zeros((nr, N), dtype=np.uint16)
    D64 = np.zeros((nr, N), dtype=np.float64) if exact else None
    rc = lib().oracle_gemm_dense(a_fmt, b_fmt, out_fmt, M, N, K, Ab.ctypes.data, Bb.ctypes.data,
                                 _ptr(Cb, ctypes.c_uint16), _ptr(r, ctypes.c_int64), nr,
                                 _ptr(D16, ctypes.c_uint16), _ptr(D64, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle: unknown element format")
    return (D16, D64) if exact else D16


def f16_to_f64(bits: int) -> float:
    return lib().oracle_f16_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return lib().oracle_bf16_to_f64(int(bits))


def e2m1_to_f64(code: int) -> float:
    return lib().oracle_e2m1_to_f64(int(code))


def e4m3_to_f64(code: int) -> float:
    return lib().oracle_e4m3_to_f64(int(code))


def e5m2_to_f64(code: int) -> float:
    return lib().oracle_e5m2_to_f64(code)


def e8m0_to_f64(code: int) -> float:
    return lib().oracle_e8m0_to_f64(int(code))


def f64_to_f16(x: float) -> int:
    return lib().oracle_f64_to_f16(float(x))


def f64_to_bf16(x: float) -> int:
    return lib().oracle_f64_to_bf16(float(x))


_F16_TABLE = None


def f16_bits_to_f64_array(bits: np.ndarray) -> np.ndarray:
    """Vector form of f16_to_f64 over a uint16 array (table over all 65536 codes)."""
    global _F16_TABLE
    if _F16_TABLE is None:
        _F16_TABLE = np.array([lib().oracle_f16_to_f64(i) for i in range(65536)],
                              dtype=np.float64)
    return _F16_TABLE[np.asarray(bits, dtype=np.uint16)]


_BF16_TABLE = None


def bf16_bits_to_f64_array(bits: np.ndarray) -> np.ndarray:
    global _BF16_TABLE
    if _BF16_TABLE is None:
        _BF16_TABLE = np.array([lib().oracle_bf16_to_f64(i) for i in range(65536)],
                               dtype=np.float64)
    return _BF16_TABLE[np.asarray(bits, dtype=np.uint16)]
