"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the CPU oracle on the same seeded bytes."""
from __future__ import annotations

import math

import numpy as np
import torch

import cute_layouts_mma_gb300 as tg
import oracle

E2M1_MAX = 6.0


def device():
    return torch.device("cuda", 0)


def to_device(prob: dict, dev) -> dict:
    out = dict(prob)
    for k in ("A", "B", "C", "SFA", "SFB"):
        if prob.get(k) is not None:
            out[k] = prob[k].to(dev)
    return out


def run_gpu(prob: dict, dev=None, accum: int = 0, D=None, stream=None):
    """Launch the CUDA GEMM for `prob` (CPU tensors) and return D on the CPU."""
    dev = dev or device()
    g = to_device(prob, dev)
    M, N = prob["M"], prob["N"]
    if prob["kind"] == "f16":
        D = torch.empty(M, N, dtype=torch.float16, device=dev) if D is None else D
        tg.gemm_f16(g["A"], g["B"], g.get("C"), D, accum, stream)
    elif prob["kind"] == "bf16":
        D = torch.empty(M, N, dtype=torch.bfloat16, device=dev) if D is None else D
        tg.gemm_bf16(g["A"], g["B"], g.get("C"), D, stream)
    elif prob["kind"] in ("fp8e4m3", "fp8e5m2"):
        fmt = tg.GEMM_FP8_E4M3 if prob["kind"] == "fp8e4m3" else tg.GEMM_FP8_E5M2
        D = torch.empty(M, N, dtype=torch.bfloat16, device=dev) if D is None else D
        tg.gemm_fp8(g["A"], g["B"], g.get("C"), D, fmt, stream)
    else:
        fmt = tg.GEMM_FMT_NVFP4 if prob["kind"] == "nvfp4" else tg.GEMM_FMT_MXFP8
        D = torch.empty(M, N, dtype=torch.bfloat16, device=dev) if D is None else D
        tg.gemm_block_scaled(g["A"], g["SFA"], g["B"], g["SFB"], g.get("C"), D, fmt, stream)
    torch.cuda.synchronize(dev)
    assert tg.gemm_last_device_error() == tg.GEMM_OK
    return D.cpu()


def oracle_result(prob: dict, rows=None):
    """(rounded output bits uint16 [rows, N], exact fp64 sums [rows, N])."""
    if prob["kind"] == "f16":
        return oracle.gemm_f16(prob["A"], prob["B"], prob.get("C"), rows=rows, exact=True)
    dense = {"bf16": oracle.BF16, "fp8e4m3": oracle.E4M3, "fp8e5m2": oracle.E5M2}
    if prob["kind"] in dense:
        f = dense[prob["kind"]]
        return oracle.gemm_dense(prob["A"], prob["B"], prob.get("C"), f, f, oracle.BF16, rows=rows, exact=True)
    fmt = oracle.NVFP4 if prob["kind"] == "nvfp4" else oracle.MXFP8
    return oracle.gemm_block_scaled(fmt, prob["A"], prob["SFA"], prob["B"], prob["SFB"],
                                    prob.get("C"), rows=rows, exact=True)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _values(t: torch.Tensor) -> np.ndarray:
    return t.double().numpy()


def operand_max(prob: dict):
    """max |a_real| and max |b_real| (bounds for the block-scaled kinds)."""
    if prob["kind"] in ("f16", "bf16"):
        return float(prob["A"].abs().max()), float(prob["B"].abs().max())
    if prob["kind"] in ("fp8e4m3", "fp8e5m2"):
        dec = oracle.e4m3_to_f64 if prob["kind"] == "fp8e4m3" else oracle.e5m2_to_f64
        mx = lambda x: max(abs(dec(int(c))) for c in torch.unique(x))
        return mx(prob["A"]), mx(prob["B"])
    if prob["kind"] == "nvfp4":
        dec = lambda sf: max(oracle.e4m3_to_f64(int(c)) for c in torch.unique(sf))
        return E2M1_MAX * dec(prob["SFA"]), E2M1_MAX * dec(prob["SFB"])
    dec_sf = lambda sf: max(oracle.e8m0_to_f64(int(c)) for c in torch.unique(sf))
    dec_x = lambda x: max(abs(oracle.e4m3_to_f64(int(c))) for c in torch.unique(x))
    return dec_x(prob["A"]) * dec_sf(prob["SFA"]), dec_x(prob["B"]) * dec_sf(prob["SFB"])


def tolerance_f32acc(prob: dict) -> float:
    """max |err| bound for fp32 accumulation: 1e-3 * sqrt(K) * max|a| * max|b|."""
    a, b = operand_max(prob)
    return 1e-3 * math.sqrt(prob["K"]) * a * b


def half_ulp(x: np.ndarray, kind: str) -> np.ndarray:
    """Half a unit in the last place of the output format at |x| (its rounding error bound)."""
    mbits, emin = (10, -14) if kind == "f16" else (7, -126)
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** emin)))
    return 0.5 * 2.0 ** (e - mbits)


def check(prob: dict, D: torch.Tensor, rows=None, mode: str = "tol", accum: int = 0) -> dict:
    """Compare the GPU output D (all rows, CPU) with the oracle.

    mode "exact": output bits identical.  mode "tol": |D - exact| <=
    1e-3*sqrt(K)*max|a|*max|b| plus half an output ulp (the output rounding,
    which the sqrt(K) term alone does not cover at small K).  mode "fro":
    relative Frobenius error <= 2e-3 (fp16 accumulation).
    """
    d16, d64 = oracle_result(prob, rows)
    got = D if rows is None else D[list(rows)]
    gbits = _bits(got)
    gval = _values(got)
    info = {"max_abs_err": float(np.max(np.abs(gval - d64))) if gval.size else 0.0}
    assert not np.isnan(gval).any(), "NaN in GPU output"
    if mode == "exact":
        bad = np.argwhere(gbits != d16)
        assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}: " \
                              f"gpu {gval[tuple(bad[0])]} oracle {d64[tuple(bad[0])]}"
    elif mode == "tol":
        tol = tolerance_f32acc(prob)
        err = np.abs(gval - d64)
        lim = tol + half_ulp(d64, prob["kind"])
        bad = np.argwhere(err > lim)
        info["tol"] = tol
        assert bad.size == 0, f"{len(bad)} outside tolerance {tol}; first {bad[:5].tolist()} " \
                              f"gpu {gval[tuple(bad[0])]} exact {d64[tuple(bad[0])]}"
    elif mode == "fro":
        rel = float(np.linalg.norm(gval - d64) / np.linalg.norm(d64))
        info["rel_fro"] = rel
        assert rel <= 2e-3, f"relative Frobenius error {rel}"
    else:
        raise ValueError(mode)
    return info


def sample_rows(M: int, n: int, seed: int = 0) -> list:
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 31, 32, 127, 128, M - 1]
    fixed = [r for r in fixed if 0 <= r < M]
    extra = rng.choice(M, size=min(M, max(0, n - len(fixed))), replace=False).tolist()
    return sorted(set(fixed + extra))


_DRIVER = {}


def dispatch_plan(M: int, N: int, K: int, kpb: int, sms: int) -> list:
    """The host-side dispatch rules' choices for one problem, from the dispatch driver
    (tests/dispatch_driver.cpp, built once per process with the host compiler):
    [fixed-scratch instance, stream-K flag, block-scaled pair, dense plan instance,
    dense plan split, block-scaled split, raster group]."""
    import os
    import shutil
    import subprocess
    import tempfile
    import pytest
    if "exe" not in _DRIVER:
        cxx = shutil.which("g++") or shutil.which("c++")
        if cxx is None:
            pytest.skip("no host C++ compiler")
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        exe = os.path.join(tempfile.mkdtemp(prefix="dispatch"), "dispatch_driver")
        subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.join(root, "cute_layouts_mma_gb300", "csrc"),
                        os.path.join(root, "tests", "dispatch_driver.cpp"), "-o", exe], check=True)
        _DRIVER["exe"] = exe
    out = subprocess.run([_DRIVER["exe"], str(sms), str(M), str(N), str(K), str(kpb)], check=True,
                         capture_output=True, text=True).stdout.split()
    return [int(v) for v in out]
