"""Key-split chunked prefill: a launch whose longest row outweighs the average load per SM
cuts long rows' key ranges into splits (partials of the softmax state) that a merge
kernel combines.  The outputs must still match the oracle on every layer kind and in both
prefill kernels (tensor-core tiles for rep * n >= 64 query rows, mma.sync below), with rows
short and long in the same launch, and the cache state stays bit-exact.
"""
import pytest

from harness import Scenario

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
def test_split_rows_all_layer_kinds(D):
    # global, sliding (W=300: the window cuts through split ranges), hybrid full + local
    sc = Scenario(B=6, max_len=4200, Hq=16, Hk=4, D=D, W=300, kinds=[0, 1, 2, 3], seed=31)
    lens = [3900, 2600, 40, 700, 0, 1500]
    while max(t - l for t, l in zip(lens, sc.lens)) > 0:
        n = [min(64, max(0, t - l)) for t, l in zip(lens, sc.lens)]
        sc.step(n, C=64, check=False)
    sc.check_state()
    # one long row among short ones; mma.sync rows (n <= 15 at rep 4) and tcgen05 rows
    sc.step([3, 64, 17, 1, 9, 40], C=64, check_state=True)
    sc.step([64, 5, 0, 33, 2, 64], C=64, check_state=True)
    sc.step([1, 1, 1, 1, 1, 1], C=1, check_state=True)


def test_split_two_query_ctas_per_row():
    """rep * n = 512 query rows: two tcgen05 CTAs per (row, kv head) share each key split."""
    sc = Scenario(B=2, max_len=3000, Hq=64, Hk=8, D=128, W=128, kinds=[0, 1], seed=32)
    sc.step([64, 10], C=64, check=False)
    while sc.lens[0] < 2800:
        sc.step([64, 0], C=64, check=False)
    sc.step([64, 64], C=64, check_state=True)
    sc.step([50, 7], C=64, check_state=True)


def test_split_paged_and_resets():
    sc = Scenario(B=4, max_len=2600, Hq=8, Hk=2, D=64, W=200, kinds=[1, 0], seed=33,
                  paged_blocks=4 * 163)
    for _ in range(36):
        sc.step([64, 64, 0, 16], C=64, check=False)
    sc.check_state()
    sc.step([20, 3, 64, 60], C=64, resets=[1], check_state=True)
    sc.step([5, 64, 1, 2], C=64, check_state=True)


def test_more_rows_than_one_launch():
    """700 rows in one call: every launch kind (append, decode, prefill, ring commit,
    state) runs in batches of at most 512 rows, on sliding, global and hybrid layers."""
    sc = Scenario(B=700, max_len=640, Hq=4, Hk=1, D=64, W=8, kinds=[1, 0, 2, 3], seed=35)
    sc.step([5] * 700, C=5, check_state=True)
    sc.step([1] * 700, C=1, check_state=True)
    rows = list(range(0, 700, 3))
    sc.step([60] * len(rows), rows=rows, C=64, check=False)
    for _ in range(8):
        sc.step([64] * len(rows), rows=rows, C=64, check=False)
    sc.check_state()
    # a mixed step over all rows: long rows (~590 keys) among short ones
    n = [(r * 7) % 40 + 1 for r in range(700)]
    sc.step(n, C=40, check_state=True)
