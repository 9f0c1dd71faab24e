"""The decode kernel against the oracle on every supported group size (1 to
8 query heads per KV head) and on context lengths around the tile and
block boundaries."""
import pytest

from paged_kv_gqa_07_gb300 import workloads as W

from _util import GpuRun, assert_close, oracle_step

pytestmark = pytest.mark.gpu

CASES = [
    ("qwen2_7b_b64", lambda: W.build(1)),
    ("tiny_qwen3", lambda: W.build(0)),
    ("g7_edges", lambda: W.custom(28, 4, ctx=[1, 15, 16, 17, 127, 128, 129, 300, 1000],
                                  q_lens=[1] * 9, seed=51)),
    ("g3", lambda: W.custom(24, 8, ctx=[5, 130, 257, 2000], q_lens=[1] * 4, seed=52)),
    ("g8", lambda: W.custom(32, 4, ctx=[64, 4096], q_lens=[1] * 2, seed=53)),
    ("g1", lambda: W.custom(8, 8, ctx=[1, 33, 128, 129, 700], q_lens=[1] * 5, seed=54)),
    ("g2", lambda: W.custom(16, 8, ctx=[2, 160, 1500], q_lens=[1] * 3, seed=55)),
    ("g4", lambda: W.custom(16, 4, ctx=[3, 511, 512, 513], q_lens=[1] * 4, seed=56)),
    ("g5", lambda: W.custom(20, 4, ctx=[90, 1025], q_lens=[1] * 2, seed=57)),
    ("g6", lambda: W.custom(24, 4, ctx=[256, 777, 31], q_lens=[1] * 3, seed=58)),
    # more sequences than the kernel keeps in shared memory (2048): context
    # lengths are read from global memory and the list is split statically
    ("b2100", lambda: W.custom(28, 4, ctx=[1 + (37 * b) % 300 for b in range(2100)],
                               q_lens=[1] * 2100, seed=59)),
    # a long list of very unequal units: runs cut through units of every size
    ("unequal", lambda: W.custom(28, 4, ctx=[4096 if b % 9 == 0 else 1 + (53 * b) % 700
                                              for b in range(200)],
                                  q_lens=[1] * 200, seed=60)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_decode_group_sizes(name, make):
    w = make()
    _, _, _, ref, e1, e2 = oracle_step(w)
    r = GpuRun(w).append().attend().sync()
    assert e1 == e2 == 0 and r.err_bits == 0, r.err_bits
    assert_close(r.out, ref)
