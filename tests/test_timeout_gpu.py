"""Failure detection on the GPU without a fault: a bounded pipeline wait runs out.

The test build of the library (compiled with TN_TIMEOUT_INJECT) withholds one
producer arrival in CTA 0, so that CTA's MMA thread waits on a stage that can
never fill.  The kernel must give up after its time limit, record the timeout,
drain its in-flight copies, free TMEM and return: the host reads
GEMM_ERR_TIMEOUT, the other CTA's tile is still computed exactly, and the CUDA
context stays usable.

The test build runs in a child process: two copies of the library (each with
its own static CUDA runtime) cannot be used in one process.  The FP16 case has
single-CTA tiles; the FP16 split case gives each tile to a cluster of CTAs; the NVFP4 case (two 128 x 128 tiles) also exercises the abandon
path of the scale issuers and scale writers; the NVFP4 pair case (40 tiles of
256 x 256, one per CTA pair) that of the CTA-pair instance.
"""
import json
import os
import subprocess
import sys
import tempfile
import textwrap

import numpy as np
import pytest
import torch

import cute_layouts_mma_gb300 as tg
from cute_layouts_mma_gb300 import build as tg_build
from cute_layouts_mma_gb300 import inputs

import _parity as P

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import ctypes, json, sys, time
    import numpy as np, torch
    sys.path.insert(0, sys.argv[1])
    from cute_layouts_mma_gb300 import build as b, inputs
    lib = ctypes.CDLL(b.build(variant="timeout_inject"))
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.gemm_f16.argtypes = [i64, i64, i64, vp, vp, vp, vp, ci, vp]
    lib.gemm_f16.restype = ci
    lib.gemm_block_scaled.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, vp, ci, vp]
    lib.gemm_block_scaled.restype = ci
    lib.gemm_last_device_error.restype = ci
    kind = sys.argv[3]
    dev = torch.device("cuda", 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if kind in ("f16", "f16split"):
        M, N, K = (128, 512, 256) if kind == "f16" else (128, 2048, 4096)
        prob = inputs.make_problem("f16", M, N, K, seed=31, dist="int2", with_c=False)
        A, B = prob["A"].to(dev), prob["B"].to(dev)
        D = torch.zeros(M, N, dtype=torch.float16, device=dev)
        torch.cuda.synchronize()
        t0 = time.time()
        rc = lib.gemm_f16(M, N, K, A.data_ptr(), B.data_ptr(), None, D.data_ptr(), 0, stream)
    else:
        M, N, K, seed = (128, 256, 512, 32) if kind == "nvfp4" else (1024, 2560, 512, 33)
        prob = inputs.make_problem("nvfp4", M, N, K, seed=seed, dist="int", with_c=False)
        g = {k: prob[k].to(dev) for k in ("A", "SFA", "B", "SFB")}
        D = torch.zeros(M, N, dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()
        t0 = time.time()
        rc = lib.gemm_block_scaled(M, N, K, g["A"].data_ptr(), g["SFA"].data_ptr(), g["B"].data_ptr(),
                                   g["SFB"].data_ptr(), None, D.data_ptr(), 0, stream)
    status = lib.gemm_last_device_error()
    elapsed = time.time() - t0
    again = lib.gemm_last_device_error()
    # the context still works after the abandoned launch
    x = torch.arange(1024, device=dev, dtype=torch.float32)
    usable = float((x * 2).sum().item()) == float(1023 * 1024)
    np.save(sys.argv[2], D.cpu().view(torch.int16).numpy())
    print(json.dumps({"rc": rc, "status": status, "again": again, "elapsed": elapsed, "usable": usable}))
""")


# (kind, the tile of the first unit: the withheld stage affects only that tile).  In
# "f16split" the first unit is CTA 0 of the first tile's cluster (128 x 2048 x 4096 FP16:
# eight 128 x 256 tiles, each split over a cluster): its CTA gives up, the cluster
# still meets at its barriers, and only that tile is affected.
CASES = [("f16", (128, 256)), ("f16split", (128, 256)), ("nvfp4", (128, 128)), ("nvfp4pair", (256, 256))]


@pytest.mark.parametrize("kind,tile0", CASES, ids=[c[0] for c in CASES])
def test_bounded_wait_runs_out_and_is_reported(kind, tile0):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    with tempfile.TemporaryDirectory() as tmp:
        script = os.path.join(tmp, "child.py")
        out_npy = os.path.join(tmp, "d.npy")
        with open(script, "w") as f:
            f.write(CHILD)
        r = subprocess.run([sys.executable, script, ROOT, out_npy, kind], capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        res = json.loads(r.stdout.strip().splitlines()[-1])
        d_bits = np.load(out_npy).view(np.uint16)
    assert res["rc"] == tg.GEMM_OK              # the launch itself was valid
    assert res["status"] == tg.GEMM_ERR_TIMEOUT  # ... and the kernel gave up and said so
    assert 1.0 <= res["elapsed"] < 60.0          # the per-wait limit is 2 s
    assert res["again"] == tg.GEMM_OK            # the record is cleared once read
    assert res["usable"]
    if kind == "f16":
        prob = inputs.make_problem("f16", 128, 512, 256, seed=31, dist="int2", with_c=False)
    elif kind == "f16split":
        prob = inputs.make_problem("f16", 128, 2048, 4096, seed=31, dist="int2", with_c=False)
    elif kind == "nvfp4":
        prob = inputs.make_problem("nvfp4", 128, 256, 512, seed=32, dist="int", with_c=False)
    else:
        prob = inputs.make_problem("nvfp4", 1024, 2560, 512, seed=33, dist="int", with_c=False)
    d16, _ = P.oracle_result(prob)
    # every other unit's tile was not affected: exact against the oracle
    other = np.ones(d16.shape, dtype=bool)
    other[:tile0[0], :tile0[1]] = False
    assert np.array_equal(d_bits[other], d16[other])
    # and this process's product library is unaffected
    P.check(prob, P.run_gpu(prob), mode="exact")
