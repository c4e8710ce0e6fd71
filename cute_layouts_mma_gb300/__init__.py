"""GB300 (sm_103a) TN matrix multiply-accumulate: Python binding of the C ABI.

The binding only marshals arguments: every step of the computation runs in the
CUDA kernels of _build/libtn_gemm.so, called through the C ABI declared in
include/tn_gemm.h.  There is no fallback: if the library cannot be built or
loaded, every call raises.

    gemm_f16(A, B, C, D, accum_dtype=GEMM_ACC_F32, stream=None)
    gemm_f16_noalloc(A, B, C, D, stream=None)
    gemm_bf16(A, B, C, D, stream=None)
    gemm_fp8(A, B, C, D, fmt, stream=None)
    gemm_block_scaled(A, SFA, B, SFB, C, D, fmt, stream=None)
    gemm_status_string(code), gemm_last_device_error()
    gemm(A, B, C=None, D=None, stream=None)   -- picks the call from A's dtype

Tensors are torch CUDA tensors used only as device memory; `stream` is a
torch.cuda.Stream (default: the current stream).
"""
from __future__ import annotations

import ctypes
import os
import threading

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_ALIGNMENT = 3
GEMM_ERR_CUDA = 4
GEMM_ERR_TIMEOUT = 5

GEMM_ACC_F32 = 0
GEMM_ACC_F16 = 1
GEMM_FMT_NVFP4 = 0
GEMM_FMT_MXFP8 = 1
GEMM_FP8_E4M3 = 0
GEMM_FP8_E5M2 = 1

EXPORTED_SYMBOLS = ("gemm_f16", "gemm_f16_noalloc", "gemm_bf16", "gemm_fp8", "gemm_block_scaled",
                    "gemm_status_string", "gemm_last_device_error")


class GemmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


_lib = None
_lock = threading.Lock()


# Test builds only (cute_layouts_mma_gb300/build.py VARIANTS): a test process may set
# TN_GEMM_TEST_VARIANT before the first call to run the same calls on a test build of
# the library, e.g. "scale_copy" (block-scaled scales moved with tcgen05.cp).
_TEST_VARIANT_ENV = "TN_GEMM_TEST_VARIANT"


def library_path() -> str:
    from . import build as _b
    return _b.lib_path(os.environ.get(_TEST_VARIANT_ENV, ""))


def lib() -> ctypes.CDLL:
    """Load the CUDA library (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                from . import build as _b
                variant = os.environ.get(_TEST_VARIANT_ENV, "")
                if variant and variant not in _b.VARIANTS:
                    raise ValueError(f"{_TEST_VARIANT_ENV}={variant!r} is not a test build of this library")
                path = _b.build(variant=variant)
                l = ctypes.CDLL(path)
                i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
                l.gemm_f16.argtypes = [i64, i64, i64, vp, vp, vp, vp, ci, vp]
                l.gemm_f16.restype = ci
                l.gemm_f16_noalloc.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp]
                l.gemm_f16_noalloc.restype = ci
                l.gemm_bf16.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp]
                l.gemm_bf16.restype = ci
                l.gemm_fp8.argtypes = [i64, i64, i64, vp, vp, vp, vp, ci, vp]
                l.gemm_fp8.restype = ci
                l.gemm_block_scaled.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, vp, ci, vp]
                l.gemm_block_scaled.restype = ci
                l.gemm_status_string.argtypes = [ci]
                l.gemm_status_string.restype = ctypes.c_char_p
                l.gemm_last_device_error.argtypes = []
                l.gemm_last_device_error.restype = ci
                _lib = l
    return _lib


def gemm_status_string(code: int) -> str:
    return lib().gemm_status_string(int(code)).decode()


def _check(code: int) -> None:
    if code != GEMM_OK:
        raise GemmError(code, gemm_status_string(code))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, shape, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gemm_f16(A, B, C, D, accum_dtype: int = GEMM_ACC_F32, stream=None) -> None:
    """D = A @ B^T + C with A half[M,K], B half[N,K], C half[M,N] or None, D half[M,N]."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    _need(A, "A", torch.float16, (M, K), dev)
    _need(B, "B", torch.float16, (N, K), dev)
    if C is not None:
        _need(C, "C", torch.float16, (M, N), dev)
    _need(D, "D", torch.float16, (M, N), dev)
    with torch.cuda.device(dev):
        _check(lib().gemm_f16(M, N, K, _ptr(A), _ptr(B), _ptr(C), _ptr(D), int(accum_dtype),
                              _stream(stream)))


def gemm_f16_noalloc(A, B, C, D, stream=None) -> None:
    """gemm_f16 with fp32 accumulation on the stream-K schedule, whose scratch is the
    library's fixed device block (no allocation).

    For callers that must not allocate device memory during the call.  Calls that
    overlap on the GPU share the block and race: keep them ordered on one stream.
    The first accepted call of the library on a device loads the block and looks up
    its address: make it before reserving the device's memory or capturing a stream.
    """
    import torch
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    _need(A, "A", torch.float16, (M, K), dev)
    _need(B, "B", torch.float16, (N, K), dev)
    if C is not None:
        _need(C, "C", torch.float16, (M, N), dev)
    _need(D, "D", torch.float16, (M, N), dev)
    with torch.cuda.device(dev):
        _check(lib().gemm_f16_noalloc(M, N, K, _ptr(A), _ptr(B), _ptr(C), _ptr(D), _stream(stream)))


def gemm_bf16(A, B, C, D, stream=None) -> None:
    """D = A @ B^T + C with A bf16[M,K], B bf16[N,K], C bf16[M,N] or None, D bf16[M,N]."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    _need(A, "A", torch.bfloat16, (M, K), dev)
    _need(B, "B", torch.bfloat16, (N, K), dev)
    if C is not None:
        _need(C, "C", torch.bfloat16, (M, N), dev)
    _need(D, "D", torch.bfloat16, (M, N), dev)
    with torch.cuda.device(dev):
        _check(lib().gemm_bf16(M, N, K, _ptr(A), _ptr(B), _ptr(C), _ptr(D), _stream(stream)))


def gemm_fp8(A, B, C, D, fmt: int, stream=None) -> None:
    """D = A @ B^T + C for FP8 A[M,K], B[N,K] (uint8 codes or float8 tensors of the
    format), C bf16[M,N] or None, D bf16[M,N]; fmt GEMM_FP8_E4M3 or GEMM_FP8_E5M2."""
    import torch
    if fmt not in (GEMM_FP8_E4M3, GEMM_FP8_E5M2):
        raise ValueError("fmt must be GEMM_FP8_E4M3 or GEMM_FP8_E5M2")
    as_u8 = lambda t: t.view(torch.uint8) if t.dtype != torch.uint8 and t.element_size() == 1 else t
    A, B = as_u8(A), as_u8(B)
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    _need(A, "A", torch.uint8, (M, K), dev)
    _need(B, "B", torch.uint8, (N, K), dev)
    if C is not None:
        _need(C, "C", torch.bfloat16, (M, N), dev)
    _need(D, "D", torch.bfloat16, (M, N), dev)
    with torch.cuda.device(dev):
        _check(lib().gemm_fp8(M, N, K, _ptr(A), _ptr(B), _ptr(C), _ptr(D), int(fmt), _stream(stream)))


def gemm_block_scaled(A, SFA, B, SFB, C, D, fmt: int, stream=None) -> None:
    """Block-scaled D = (A*SFA) @ (B*SFB)^T + C; operands as uint8, C/D bf16[M,N].

    NVFP4: A uint8[M, K/2] (two E2M1 codes per byte, low nibble first), SFA uint8[M, K/16] E4M3.
    MXFP8: A uint8[M, K] (E4M3 codes; float8_e4m3fn tensors are accepted), SFA uint8[M, K/32] E8M0.
    """
    import torch
    as_u8 = lambda t: t.view(torch.uint8) if t is not None and t.dtype != torch.uint8 and t.element_size() == 1 else t
    A, B, SFA, SFB = as_u8(A), as_u8(B), as_u8(SFA), as_u8(SFB)
    M = A.shape[0]
    N = B.shape[0]
    if fmt == GEMM_FMT_NVFP4:
        K, kblk = A.shape[1] * 2, 16
    elif fmt == GEMM_FMT_MXFP8:
        K, kblk = A.shape[1], 32
    else:
        raise ValueError("fmt must be GEMM_FMT_NVFP4 or GEMM_FMT_MXFP8")
    dev = A.device
    _need(A, "A", torch.uint8, A.shape, dev)
    _need(B, "B", torch.uint8, (N, A.shape[1]), dev)
    _need(SFA, "SFA", torch.uint8, (M, K // kblk), dev)
    _need(SFB, "SFB", torch.uint8, (N, K // kblk), dev)
    if C is not None:
        _need(C, "C", torch.bfloat16, (M, N), dev)
    _need(D, "D", torch.bfloat16, (M, N), dev)
    with torch.cuda.device(dev):
        _check(lib().gemm_block_scaled(M, N, K, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C),
                                       _ptr(D), int(fmt), _stream(stream)))


def gemm_last_device_error() -> int:
    """Synchronise the current device; GEMM_ERR_TIMEOUT if a kernel abandoned its work."""
    return lib().gemm_last_device_error()


def gemm(A, B, C=None, D=None, stream=None, accum_dtype: int = GEMM_ACC_F32):
    """D = A @ B^T + C, choosing the call from A's dtype: float16 -> gemm_f16 (fp16 D),
    bfloat16 -> gemm_bf16, float8_e4m3fn / float8_e5m2 -> gemm_fp8 (bf16 D).  D is
    allocated when not given; it is returned.  Block-scaled operands need their scale
    tensors: use gemm_block_scaled for those."""
    import torch
    M, N = A.shape[0], B.shape[0]
    kinds = {torch.float16: torch.float16, torch.bfloat16: torch.bfloat16,
             torch.float8_e4m3fn: torch.bfloat16, torch.float8_e5m2: torch.bfloat16}
    if A.dtype not in kinds:
        raise ValueError(f"unsupported operand dtype {A.dtype}")
    if D is None:
        D = torch.empty(M, N, dtype=kinds[A.dtype], device=A.device)
    if A.dtype == torch.float16:
        gemm_f16(A, B, C, D, accum_dtype, stream)
    elif A.dtype == torch.bfloat16:
        gemm_bf16(A, B, C, D, stream)
    else:
        if B.dtype != A.dtype:
            raise ValueError("A and B must have the same FP8 format")
        gemm_fp8(A, B, C, D, GEMM_FP8_E4M3 if A.dtype == torch.float8_e4m3fn else GEMM_FP8_E5M2, stream)
    return D

