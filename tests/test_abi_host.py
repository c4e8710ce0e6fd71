"""The C-ABI library loads, exports every symbol include/tn_gemm.h declares, and
rejects bad arguments on the host before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest
import torch

import cute_layouts_mma_gb300 as tg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                            src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    assert set(_declared_functions()) == set(tg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = tg.lib()
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings():
    for code in range(6):
        s = tg.gemm_status_string(code)
        assert s.startswith("GEMM_")
    assert "unknown" in tg.gemm_status_string(99)


P = 1 << 20  # fake, 16-byte aligned "device" addresses: never dereferenced on rejection


def _f16(M, N, K, A=P, B=2 * P, C=None, D=4 * P, acc=0):
    return tg.lib().gemm_f16(M, N, K, A, B, C, D, acc, None)


def _bs(M, N, K, fmt, A=P, SFA=2 * P, B=3 * P, SFB=4 * P, C=None, D=6 * P):
    return tg.lib().gemm_block_scaled(M, N, K, A, SFA, B, SFB, C, D, fmt, None)


def test_f16_rejections():
    assert _f16(0, 8, 8) == tg.GEMM_ERR_INVALID_ARG
    assert _f16(8, -8, 8) == tg.GEMM_ERR_INVALID_ARG
    assert _f16(1 << 31, 8, 8) == tg.GEMM_ERR_INVALID_ARG
    assert _f16(8, 8, 8, A=None) == tg.GEMM_ERR_INVALID_ARG
    assert _f16(8, 8, 8, D=None) == tg.GEMM_ERR_INVALID_ARG
    assert _f16(8, 8, 8, acc=2) == tg.GEMM_ERR_INVALID_ARG
    assert _f16(8, 8, 12) == tg.GEMM_ERR_ALIGNMENT          # K % 8
    assert _f16(8, 12, 8) == tg.GEMM_ERR_ALIGNMENT          # N % 8
    assert _f16(8, 8, 8, A=P + 8) == tg.GEMM_ERR_ALIGNMENT  # pointer alignment
    assert _f16(8, 8, 8, C=P + 2) == tg.GEMM_ERR_ALIGNMENT
    # D overlapping A or B, or partially overlapping C
    assert _f16(64, 64, 64, D=P + 16) == tg.GEMM_ERR_INVALID_ARG
    assert _f16(64, 64, 64, D=2 * P) == tg.GEMM_ERR_INVALID_ARG
    assert _f16(64, 64, 64, C=4 * P + 16) == tg.GEMM_ERR_INVALID_ARG


def test_f16_noalloc_rejections():
    f = lambda M, N, K, A=P, B=2 * P, C=None, D=4 * P: tg.lib().gemm_f16_noalloc(M, N, K, A, B, C, D, None)
    assert f(0, 8, 8) == tg.GEMM_ERR_INVALID_ARG
    assert f(8, 8, 8, B=None) == tg.GEMM_ERR_INVALID_ARG
    assert f(8, 8, 12) == tg.GEMM_ERR_ALIGNMENT
    assert f(8, 8, 8, D=P + 8) == tg.GEMM_ERR_ALIGNMENT
    assert f(64, 64, 64, D=2 * P) == tg.GEMM_ERR_INVALID_ARG


def test_bf16_and_fp8_rejections():
    bf = lambda M, N, K, A=P, B=2 * P, C=None, D=4 * P: tg.lib().gemm_bf16(M, N, K, A, B, C, D, None)
    f8 = lambda M, N, K, fmt=0, A=P, B=2 * P, C=None, D=4 * P: tg.lib().gemm_fp8(M, N, K, A, B, C, D, fmt, None)
    assert bf(0, 8, 8) == tg.GEMM_ERR_INVALID_ARG
    assert bf(8, 8, 12) == tg.GEMM_ERR_ALIGNMENT          # K % 8
    assert bf(8, 12, 8) == tg.GEMM_ERR_ALIGNMENT          # N % 8
    assert bf(64, 64, 64, D=2 * P) == tg.GEMM_ERR_INVALID_ARG
    assert f8(8, 8, 16, fmt=2) == tg.GEMM_ERR_INVALID_ARG
    assert f8(8, 8, 8) == tg.GEMM_ERR_ALIGNMENT           # K % 16 (16-byte rows)
    assert f8(8, 8, 16, A=None) == tg.GEMM_ERR_INVALID_ARG
    assert f8(64, 64, 64, C=4 * P + 16) == tg.GEMM_ERR_INVALID_ARG


def test_block_scaled_rejections():
    for fmt in (tg.GEMM_FMT_NVFP4, tg.GEMM_FMT_MXFP8):
        assert _bs(0, 8, 512, fmt) == tg.GEMM_ERR_INVALID_ARG
        assert _bs(8, 8, 512, fmt, SFA=None) == tg.GEMM_ERR_INVALID_ARG
        assert _bs(8, 8, 512, fmt, D=P) == tg.GEMM_ERR_INVALID_ARG  # D == A
        assert _bs(8, 12, 512, fmt) == tg.GEMM_ERR_ALIGNMENT
        assert _bs(8, 8, 512, fmt, SFB=4 * P + 4) == tg.GEMM_ERR_ALIGNMENT
    assert _bs(8, 8, 512, 2) == tg.GEMM_ERR_INVALID_ARG
    assert _bs(8, 8, 8, tg.GEMM_FMT_NVFP4) == tg.GEMM_ERR_INVALID_ARG    # not whole blocks of 16
    assert _bs(8, 8, 48, tg.GEMM_FMT_MXFP8) == tg.GEMM_ERR_INVALID_ARG   # not whole blocks of 32
    assert _bs(8, 8, 128, tg.GEMM_FMT_NVFP4) == tg.GEMM_ERR_ALIGNMENT    # scale row 8 bytes
    assert _bs(8, 8, 256, tg.GEMM_FMT_MXFP8) == tg.GEMM_ERR_ALIGNMENT    # scale row 8 bytes


def test_valid_call_without_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _f16(8, 8, 8) in (tg.GEMM_ERR_CUDA, tg.GEMM_ERR_UNSUPPORTED)
    assert _bs(8, 8, 256, tg.GEMM_FMT_NVFP4) in (tg.GEMM_ERR_CUDA, tg.GEMM_ERR_UNSUPPORTED)


def test_python_wrappers_check_arguments_before_the_library():
    # dtype, shape, device and layout checks happen in the binding (CPU tensors here)
    A = torch.zeros(8, 16, dtype=torch.float16)
    with pytest.raises(ValueError):
        tg.gemm_f16(A, A, None, torch.zeros(8, 8, dtype=torch.float16))       # not CUDA tensors
    with pytest.raises(ValueError):
        tg.gemm_bf16(A, A, None, torch.zeros(8, 8, dtype=torch.bfloat16))     # A is not bf16
    with pytest.raises(ValueError):
        tg.gemm_fp8(A.view(torch.uint8), A.view(torch.uint8), None, torch.zeros(8, 8), 5)  # unknown format
    with pytest.raises(ValueError):
        tg.gemm_block_scaled(A.view(torch.uint8), None, A.view(torch.uint8), None, None,
                             torch.zeros(8, 8, dtype=torch.bfloat16), 7)       # unknown format
