"""The pages' scale-copy instruction as a tested compile-time alternative.

The block-scaled kernels place the scale factors in TMEM with tcgen05.st from four
writer warps (the product path).  The test build "scale_copy" (TN_SCALE_COPY) instead
repacks each stage's scales in shared memory into the 32-lane x 16-byte base tiles of
"数据布局及其记号" (section on TMEM scale factors: local_lane = m % 32, TCol = m // 32,
byte = sfk) and copies them with tcgen05.cp.32x128b.warpx4, which replicates the tile
to the four lane partitions.  This runs the block-scaled parity tests (integer inputs
bit-exact against the oracle, the one-hot scale probes, ragged shapes, CTA pairs and
cluster splits) on that build, in a child process: two copies of the library (each
with its own static CUDA runtime) cannot be used in one process.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SELECT = ("one_hot or nvfp4_integers or mxfp8_integers or block_scaled_pair or nvfp4_random or mxfp8_random "
          "or split_nvfp4 or split_mxfp8 or large_k_nvfp4")


def test_block_scaled_parity_with_scale_copies():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, TN_GEMM_TEST_VARIANT="scale_copy")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gemm_gpu.py"), "-m", "gpu",
                        "-q", "-x", "-k", SELECT, "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
