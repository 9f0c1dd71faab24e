"""Both decode kernels against the oracle: the tensor-core kernel (the
default) and the CUDA-core kernel, each selected in a fresh process through
QATTN_DECODE_KERNEL, on group sizes 1 to 8."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

SCRIPT = r"""
import sys
sys.path.insert(0, {here!r})
sys.path.insert(0, {root!r})
from paged_kv_gqa_07_gb300 import workloads as W
from _util import GpuRun, assert_close, oracle_step
cases = [W.build(1), W.build(0),
         W.custom(28, 4, ctx=[1, 15, 16, 17, 127, 128, 129, 300, 1000], q_lens=[1] * 9, seed=51),
         W.custom(24, 8, ctx=[5, 130, 257, 2000], q_lens=[1] * 4, seed=52),
         W.custom(32, 4, ctx=[64, 4096], q_lens=[1] * 2, seed=53),
         W.custom(8, 8, ctx=[1, 33, 128, 129, 700], q_lens=[1] * 5, seed=54),
         W.custom(16, 8, ctx=[2, 160, 1500], q_lens=[1] * 3, seed=55)]
for w in cases:
    _, _, _, ref, _, _ = oracle_step(w)
    r = GpuRun(w).append().attend().sync()
    assert r.err_bits == 0, r.err_bits
    mx, rel = assert_close(r.out, ref)
    print(w.name, w.num_heads // w.num_kv_heads, "max abs %.3e" % mx)
print("ok")
"""


@pytest.mark.parametrize("kernel", ["tc", "cuda"])
def test_decode_kernel_forced(kernel):
    env = dict(os.environ, QATTN_DECODE_KERNEL=kernel)
    code = SCRIPT.format(here=HERE, root=os.path.dirname(HERE))
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout + res.stderr
